"""Phase timeline of the tile kernels over a sequence of calls (a diagnostic).

    python -m nvfp4_weight_only_gemv_gb300.phase_trace [--steps S] [--no-pdl] CALL [CALL ...]

CALL is ``dense:N:K:M[:bf16]``, ``gate_up:N:K:M``, ``swiglu:N:K:M``, ``ffn:H:I:M`` (the FFN block
in one call) or ``moe:E:N:K:T:TOPK:XPS`` (XPS 1: one x row per slot). The library is rebuilt with ``-DNVFP4_PHASE_TRACE=1`` into its own
file and loaded instead of the normal build. The calls of a step run back to back behind a
sleep kernel, as bench.py times them, with weight copies rotating through more than twice the
L2, for a few warm-up steps and then S traced steps (S * calls <= 16, the trace's launch slots).

For every traced launch it prints, in microseconds from the first CTA entry of the traced
steps: when the launch's CTAs entered (first, median, last), when they were past the
dependency wait, when x was staged, when the first weight box landed, when the outputs were
stored and when the last CTA exited; then each launch's share of the chain (last exit minus
the previous launch's last exit) and its algorithmic bytes over that time.
"""
from __future__ import annotations

import argparse
import math
import os
import sys

import numpy as np
import torch

from . import build as _build

PHASES = ["entry", "issued", "dep_wait", "x_staged", "first_box", "loop_done", "stored", "exit"]


def parse_call(spec: str):
    f = spec.split(":")
    kind = f[0]
    if kind in ("dense", "gate_up", "swiglu", "ffn"):
        N, K, M = (int(v) for v in f[1:4])
        bf16 = len(f) > 4 and f[4] == "bf16"
        return {"kind": kind, "N": N, "K": K, "M": M, "bf16": bf16}
    if kind == "moe":
        E, N, K, T, top_k, xps = (int(v) for v in f[1:7])
        return {"kind": kind, "E": E, "N": N, "K": K, "T": T, "top_k": top_k, "xps": bool(xps), "bf16": False}
    raise SystemExit(f"bad call spec {spec!r}")


def make_sets(c, copies, seed, dev):
    from . import synth
    sets = []
    if c["kind"] == "dense":
        base = synth.dense_problem(c["N"], c["K"], c["M"], seed, device=dev)
    elif c["kind"] in ("gate_up", "swiglu"):
        base = synth.gate_up_problem(c["N"], c["K"], c["M"], seed, device=dev)
    elif c["kind"] == "ffn":
        base = synth.ffn_problem(c["N"], c["K"], c["M"], seed, device=dev)
    else:
        base = synth.moe_problem(c["E"], c["N"], c["K"], c["T"], c["top_k"], c["xps"], seed=seed, device=dev,
                                  fill="all")
    for i in range(copies):
        d = {k: (v.clone() if isinstance(v, torch.Tensor) and (i == 0 or c["kind"] != "moe") else v)
             for k, v in base.items()}
        if c["kind"] == "moe" and i > 0:
            d = dict(sets[0])
            d["ids"] = synth.routing(c["T"], c["top_k"], c["E"], seed * 7919 + i).to(dev)
        if c["kind"] == "ffn":
            import nvfp4_weight_only_gemv_gb300 as nv
            d["ws"] = nv.ffn_workspace(c["M"], c["K"], dev)
        sets.append(d)
    return sets


def weight_bytes(c, d):
    per_row = c["K"] * 0.5 + c["K"] / 16
    if c["kind"] in ("gate_up", "swiglu"):
        return 2 * c["N"] * per_row
    if c["kind"] == "ffn":
        return 3 * c["N"] * per_row  # gate and up [I, H], down [H, I]: 3 * H * I weights
    if c["kind"] == "moe":
        return len(set(d["ids"].tolist())) * c["N"] * per_row
    return c["N"] * per_row


def alg_bytes(c, d):
    ob = 2 if c["bf16"] else 4
    if c["kind"] == "moe":
        slots = c["T"] * c["top_k"]
        xr = slots if c["xps"] else c["T"]
        return weight_bytes(c, d) + xr * c["K"] * 2 + slots * c["N"] * ob
    if c["kind"] == "ffn":  # x [M, H] in, y [M, H] out (h stays inside the call)
        return weight_bytes(c, d) + c["M"] * c["N"] * (2 + ob)
    cols = c["N"] * (2 if c["kind"] == "gate_up" else 1)
    return weight_bytes(c, d) + c["M"] * c["K"] * 2 + c["M"] * cols * ob


def launch(nv, c, d, x=None):
    """One call; x replaces the call's own x (chained mode). Returns y."""
    dt = torch.bfloat16 if c["bf16"] else torch.float32
    x = d["x"] if x is None else x
    if c["kind"] == "dense":
        return nv.gemv(d["w"], d["s"], d["g"], x, out_dtype=dt)
    if c["kind"] == "gate_up":
        return nv.gemv_gate_up(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], x, out_dtype=dt)
    if c["kind"] == "swiglu":
        return nv.gemv_gate_up_swiglu(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], x, 10.0, out_dtype=dt)
    if c["kind"] == "ffn":
        return nv.ffn_swiglu(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], d["wd"], d["sd"], d["gd"], x,
                             10.0, workspace=d["ws"], out_dtype=dt)
    return nv.moe_gemv(d["w"], d["s"], d["gs"], d["ids"], x, c["xps"], c["top_k"], out_dtype=dt)


def summarise(tr, launches, calls_meta):
    """tr: [16, 1024, 40] int64. Returns the report lines."""
    tr = tr.numpy().astype(np.int64)
    entries = tr[:launches, :, 0]
    origin = entries[entries > 0].min()
    us = lambda v: (v - origin) / 1e3
    lines = []
    hdr = (f"{'launch':<28}{'ctas':>5}{'entry first/med/last':>24}{'dep_wait med/last':>20}{'x_staged med':>14}"
           f"{'1st_box med':>13}{'stored med/last':>18}{'exit last':>11}{'chain us':>10}{'GB/s':>8}")
    lines.append(hdr)
    prev_exit = None
    for l in range(launches):
        rows = tr[l][tr[l, :, 0] > 0]
        name, nbytes = calls_meta[l]
        if len(rows) == 0:
            lines.append(f"{name:<28} (not traced)")
            continue
        ph = lambda p: rows[:, 2 * p][rows[:, 2 * p] > 0]
        def med(p):
            v = ph(p)
            return f"{us(np.median(v)):.2f}" if len(v) else "-"
        def last(p):
            v = ph(p)
            return f"{us(v.max()):.2f}" if len(v) else "-"
        e = ph(0)
        ex = ph(7).max()
        chain = us(ex) - (us(prev_exit) if prev_exit is not None else us(e.min()))
        prev_exit = ex
        lines.append(f"{name:<28}{len(rows):>5}{us(e.min()):>8.2f}/{us(np.median(e)):.2f}/{us(e.max()):.2f}"
                     f"{med(2) + '/' + last(2):>20}{med(3):>14}{med(4):>13}{med(6) + '/' + last(6):>18}"
                     f"{us(ex):>11.2f}{chain:>10.2f}{nbytes / (chain * 1e-6) / 1e9 if chain > 0 else 0:>8.0f}")
    # per-CTA phase durations (median over all traced CTAs of each launch)
    lines.append("")
    lines.append(f"{'launch':<28}" + "".join(f"{a + '->' + b:>20}" for a, b in
                                             [("entry", "dep_wait"), ("dep_wait", "x_staged"),
                                              ("x_staged", "first_box"), ("first_box", "stored"),
                                              ("stored", "exit")]) + f"{'SM GHz':>8}")
    for l in range(launches):
        rows = tr[l][tr[l, :, 0] > 0]
        if len(rows) == 0:
            continue
        def d(a, b):
            ok = (rows[:, 2 * a] > 0) & (rows[:, 2 * b] > 0)
            return f"{np.median(rows[ok, 2 * b] - rows[ok, 2 * a]) / 1e3:.2f}" if ok.any() else "-"
        ok = (rows[:, 14] > 0) & (rows[:, 0] > 0) & (rows[:, 14] > rows[:, 0])
        ghz = np.median((rows[ok, 15] - rows[ok, 1]) / (rows[ok, 14] - rows[ok, 0])) if ok.any() else float("nan")
        lines.append(f"{calls_meta[l][0]:<28}{d(0, 2):>20}{d(2, 3):>20}{d(3, 4):>20}{d(4, 6):>20}{d(6, 7):>20}"
                     f"{ghz:>8.2f}")
    # per-warp spread inside a CTA: first box landed and box loop left, relative to x staged
    lines.append("")
    lines.append(f"{'launch':<28}{'1st box: warp med/max after x_staged':>38}{'loop end: warp med/max after x_staged':>40}")
    for l in range(launches):
        rows = tr[l][tr[l, :, 0] > 0]
        if len(rows) == 0:
            continue
        first = np.concatenate([rows[:, 8:9], rows[:, 25:32]], axis=1).astype(np.float64)
        loop = rows[:, 16:24].astype(np.float64)
        xs = rows[:, 6:7].astype(np.float64)
        def stat(a):
            ok = (a > 0) & (xs > 0)
            d = np.where(ok, a - xs, np.nan)
            return f"{np.nanmedian(d) / 1e3:.2f}/{np.nanmax(d) / 1e3:.2f}" if ok.any() else "-"
        lines.append(f"{calls_meta[l][0]:<28}{stat(first):>38}{stat(loop):>40}")
    # the tail: when CTAs stored their outputs (phase 6) relative to the launch's median, and the
    # SMs (word 24) of the last four
    lines.append("")
    lines.append(f"{'launch':<28}{'stored p90-med (us)':>22}{'stored last-med (us)':>22}{'SMs of the last 4 CTAs':>30}")
    for l in range(launches):
        rows = tr[l][tr[l, :, 0] > 0]
        st = rows[:, 12]
        ok = st > 0
        if ok.sum() < 4:
            continue
        med = np.median(st[ok])
        last4 = np.argsort(np.where(ok, st, 0))[-4:]
        lines.append(f"{calls_meta[l][0]:<28}{(np.percentile(st[ok], 90) - med) / 1e3:>22.2f}"
                     f"{(st[ok].max() - med) / 1e3:>22.2f}{' '.join(str(int(rows[i, 24])) for i in last4):>30}")
    # dense launches, thread 0 in SM cycles: x staged (phase 3's clock) to just before the wait
    # for its first box (word 38), and that wait (word 38 to 39)
    dense = [l for l in range(launches) if calls_meta[l][0].startswith(("dense", "gate_up", "swiglu"))]
    if dense:
        lines.append("")
        lines.append(f"{'launch':<28}{'x_staged->box wait (cycles)':>30}{'box wait (cycles)':>20}"
                     f"{'issued->landed (us)':>22}{'landed->dep_wait (us)':>24}")
        for l in dense:
            rows = tr[l][tr[l, :, 0] > 0]
            ok = (rows[:, 7] > 0) & (rows[:, 38] > 0) & (rows[:, 39] > 0)
            if not ok.any():
                continue
            r = rows[ok]
            # word 36: when the first box landed (builds with NVFP4_TRACE_BOX_LANDED=1 only)
            land = r[r[:, 36] > 0]
            il = f"{np.median(land[:, 36] - land[:, 2]) / 1e3:.2f}" if len(land) else "-"
            ld = f"{np.median(land[:, 4] - land[:, 36]) / 1e3:.2f}" if len(land) else "-"
            lines.append(f"{calls_meta[l][0]:<28}{np.median(r[:, 38] - r[:, 7]):>30.0f}"
                         f"{np.median(r[:, 39] - r[:, 38]):>20.0f}{il:>22}{ld:>24}")
    # the FFN block's own phases (thread 0, so warp 0's K slice): gate/up done (phase 5), its
    # slice of h complete (word 38), that slice staged (word 39), down done (phase 6)
    ffn = [l for l in range(launches) if calls_meta[l][0].startswith("ffn")]
    if ffn:
        lines.append("")
        lines.append(f"{'launch':<28}" + "".join(f"{h:>20}" for h in
                                                 ("x_staged->gu_done", "gu_done->slice_ready",
                                                  "ready->h_staged", "h_staged->down_done", "ready last-first")))
        for l in ffn:
            rows = tr[l][tr[l, :, 0] > 0]
            def dd(a, b):
                ok = (a > 0) & (b > 0)
                return f"{np.median(b[ok] - a[ok]) / 1e3:.2f}" if ok.any() else "-"
            bar = rows[:, 38][rows[:, 38] > 0]
            spread = f"{(bar.max() - bar.min()) / 1e3:.2f}" if len(bar) else "-"
            lines.append(f"{calls_meta[l][0]:<28}{dd(rows[:, 6], rows[:, 10]):>20}{dd(rows[:, 10], rows[:, 38]):>20}"
                         f"{dd(rows[:, 38], rows[:, 39]):>20}{dd(rows[:, 39], rows[:, 12]):>20}{spread:>20}")
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("calls", nargs="+")
    ap.add_argument("--steps", type=int, default=0, help="traced steps (default: as many as fit 16 launches)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--define", action="append", default=[], help="extra NAME=VALUE for the traced build")
    ap.add_argument("--save", default=None, help="also write the raw trace of the traced launches (.npy)")
    ap.add_argument("--chain", action="store_true",
                    help="each call's x is the previous call's output (dense bf16 calls with N = next K and equal M)")
    args = ap.parse_args(argv)
    calls = [parse_call(s) for s in args.calls]
    steps = args.steps or max(1, 16 // len(calls))
    if steps * len(calls) > 16:
        raise SystemExit("steps * calls must be <= 16 (the trace's launch slots)")
    defines = {"NVFP4_PHASE_TRACE": 1}
    for kv in args.define:
        k, v = kv.split("=", 1)
        defines[k] = v
    name = "trace" + "".join(f"_{k.lower()}{v}" for k, v in sorted(defines.items()) if k != "NVFP4_PHASE_TRACE")
    os.environ["NVFP4_GEMV_LIBRARY"] = _build.build_variant(name, defines)
    import nvfp4_weight_only_gemv_gb300 as nv
    nv.library()
    if args.no_pdl:
        nv.set_pdl(False)
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    step_w = 0
    for c in calls:
        rows = c["N"] * {"gate_up": 2, "swiglu": 2, "ffn": 3}.get(c["kind"], 1)
        step_w += 0 if c["kind"] == "moe" else rows * c["K"] * 9 // 16
    copies = max(steps + 1, math.ceil(2.5 * l2 / step_w)) if step_w else 4
    sets = [make_sets(c, copies, 11 + i, dev) for i, c in enumerate(calls)]
    if args.chain:
        for a, b in zip(calls, calls[1:] + calls[:1]):
            if not (a["kind"] == b["kind"] == "dense" and a["bf16"] and a["N"] == b["K"] and a["M"] == b["M"]):
                raise SystemExit("--chain needs dense bf16 calls with N equal to the next call's K")

    def step(k):
        y = None
        for ci, c in enumerate(calls):
            y = launch(nv, c, sets[ci][k % copies], x=y if args.chain else None)

    k = 0
    for _ in range(args.warmup):
        step(k)
        k += 1
    torch.cuda.synchronize()
    nv.phase_trace()  # clear; restart the slots
    meta = [(args.calls[ci][:27], alg_bytes(c, sets[ci][(k + st) % copies]))  # host work before the launches
            for st in range(steps) for ci, c in enumerate(calls)]
    torch.cuda._sleep(int(2e6))  # the launches queue up behind it, so the GPU sees them back to back
    for _ in range(steps):
        step(k)
        k += 1
    tr = nv.phase_trace()
    if tr is None:
        raise SystemExit("the loaded library was built without the phase trace")
    if args.save:
        np.save(args.save, tr[:len(meta)].numpy())
    flags = nv.device_status()
    print(f"# {props.name}, {props.multi_processor_count} SMs; PDL {'off' if args.no_pdl else 'on'}; "
          f"x {'chained (previous output)' if args.chain else 'per call'}; "
          f"{steps} traced step(s) of {len(calls)} call(s); build defines {defines}; device status {flags}")
    for c in calls:
        kind = {"swiglu": "gate_up_swiglu", "moe": "moe_per_slot" if c.get("xps") else "moe"}.get(c["kind"], c["kind"])
        if c["kind"] == "moe":
            print("#", nv.describe_plan(kind, c["E"], c["N"], c["K"], c["T"], c["top_k"]))
        else:
            print("#", nv.describe_plan(kind, c["M"], c["N"], c["K"]))
    print("\n".join(summarise(tr, len(meta), meta)))
    return 0


if __name__ == "__main__":
    sys.exit(main())
