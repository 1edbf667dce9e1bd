"""DRAM traffic and occupancy of the library's kernels per bench workload, measured with ncu.

    python -m nvfp4_weight_only_gemv_gb300.ncu_traffic [--workloads vocab,attn,...] [--out DIR]

For every workload it first runs ``bench.py --workload W`` plainly (it must exit 0), then the
same command under ncu with ``--clock-control none``, capturing the launches of one timed step
of the library's kernels (``-k regex:gemv_``, after the warm-up launches) with these counters:

  gpu__time_duration.sum                                   launch time (cold, serialised)
  dram__bytes_read.sum, dram__bytes_write.sum               DRAM traffic per launch
  l1tex__t_sectors_pipe_lsu_mem_global_op_ld.sum,
  l1tex__t_requests_pipe_lsu_mem_global_op_ld.sum           sectors per request of global loads
                                                            (x staging; weights arrive by TMA)
  sm__warps_active.avg.pct_of_peak_sustained_active         achieved occupancy

It writes ``traffic.json`` (per workload: DRAM read + write bytes per launch, averaged over the
captured launches, tied to the sha256 of the kernel source it measured; bench.py reports it as
``roofline.traffic`` only while the source is unchanged) and ``counters.md`` (a table of every
captured launch) into DIR (default: the package's _build/ncu_traffic). The raw CSVs stay in DIR.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "nvfp4_weight_only_gemv_gb300", "csrc", "nvfp4_gemv.cu")

METRICS = ["gpu__time_duration.sum", "dram__bytes_read.sum", "dram__bytes_write.sum",
           "l1tex__t_sectors_pipe_lsu_mem_global_op_ld.sum", "l1tex__t_requests_pipe_lsu_mem_global_op_ld.sum",
           "sm__warps_active.avg.pct_of_peak_sustained_active"]
# launches of one step of each workload (captured after the warm-up launches)
LAUNCHES = {"vocab": 1, "vocab_sdict": 1, "attn": 4, "ffn": 2, "ffn_m2": 2, "ffn_m4": 2, "ffn_m8": 2, "ffn_swiglu": 2,
            "ffn_fused": 2, "ffn_shared": 2, "ffn_shared_fused": 1, "moe": 2, "moe_sdict": 2, "moe_t32": 2,
            "card_m2": 5}
WARMUP = 3


def source_sha256() -> str:
    with open(SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def bench_cmd(workload: str):
    return [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", workload, "--steps", "2",
            "--warmup", str(WARMUP), "--no-cpu-baseline", "--no-per-workload"]


def parse(csv_text: str):
    """Rows of ncu's --csv --page raw output: [{'Kernel Name': ..., metric: value}, ...]."""
    lines = [l for l in csv_text.splitlines() if l.startswith('"')]
    if not lines:
        return []
    rows = list(csv.DictReader(io.StringIO("\n".join(lines))))
    out = []
    for r in rows:
        if not r.get("ID", "").strip().isdigit():
            continue  # the units row
        rec = {"kernel": r.get("Kernel Name", ""), "id": int(r["ID"])}
        for m in METRICS:
            v = r.get(m, "").replace(",", "")
            try:
                rec[m] = float(v)
            except ValueError:
                rec[m] = None
        out.append(rec)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workloads", default="vocab,attn,card_m2,ffn,ffn_m2,ffn_m4,ffn_m8,ffn_swiglu,ffn_fused,"
                                           "ffn_shared,ffn_shared_fused,moe,moe_t32,vocab_sdict,moe_sdict")
    ap.add_argument("--out", default=os.path.join(ROOT, "nvfp4_weight_only_gemv_gb300", "_build", "ncu_traffic"))
    args = ap.parse_args(argv)
    os.makedirs(args.out, exist_ok=True)
    sha = source_sha256()
    per_launch, table = {}, []
    for w in args.workloads.split(","):
        plain = subprocess.run(bench_cmd(w), capture_output=True, text=True, timeout=900)
        if plain.returncode != 0:
            print(f"{w}: plain run failed (rc {plain.returncode}); not profiled", flush=True)
            continue
        n = LAUNCHES.get(w, 2)
        log = os.path.join(args.out, f"{w}.csv")
        cmd = ["ncu", "--clock-control", "none", "--metrics", ",".join(METRICS), "-k", "regex:gemv_",
               "-s", str(WARMUP * n), "-c", str(n), "--csv", "--page", "raw", "--log-file", log] + bench_cmd(w)
        res = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
        if res.returncode != 0 or not os.path.exists(log):
            print(f"{w}: ncu rc {res.returncode}", flush=True)
            continue
        rows = parse(open(log).read())
        if not rows:
            print(f"{w}: no launches captured", flush=True)
            continue
        traffic = [r["dram__bytes_read.sum"] + r["dram__bytes_write.sum"] for r in rows
                   if r["dram__bytes_read.sum"] is not None and r["dram__bytes_write.sum"] is not None]
        per_launch[w] = int(round(sum(traffic) / len(traffic))) if traffic else None
        for r in rows:
            sec, req = r["l1tex__t_sectors_pipe_lsu_mem_global_op_ld.sum"], r["l1tex__t_requests_pipe_lsu_mem_global_op_ld.sum"]
            table.append((w, r["kernel"].split("(")[0], r["gpu__time_duration.sum"], r["dram__bytes_read.sum"],
                          r["dram__bytes_write.sum"], (sec / req) if sec and req else None,
                          r["sm__warps_active.avg.pct_of_peak_sustained_active"]))
        print(f"{w}: {len(rows)} launches, {per_launch[w]} DRAM bytes per launch", flush=True)
    rec = {"kernel_source_sha256": sha,
           "how": "python -m nvfp4_weight_only_gemv_gb300.ncu_traffic: ncu --clock-control none --metrics "
                  + ",".join(METRICS) + " on one timed step of bench.py --workload W (after its warm-up "
                  "launches); dram__bytes_read.sum + dram__bytes_write.sum averaged over the step's launches",
           "dram_bytes_per_launch": per_launch}
    with open(os.path.join(args.out, "traffic.json"), "w") as f:
        json.dump(rec, f, indent=2)
    with open(os.path.join(args.out, "counters.md"), "w") as f:
        f.write("| workload | kernel | time (us, ncu) | DRAM read (MB) | DRAM write (MB) | sectors/request (LSU loads) "
                "| warps active (% of peak) |\n|---|---|---|---|---|---|---|\n")
        for w, k, t, rd, wr, spr, occ in table:
            fmt = lambda v, s, d=2: "-" if v is None else f"{v / s:.{d}f}"
            f.write(f"| {w} | {k} | {fmt(t, 1e3)} | {fmt(rd, 1e6)} | {fmt(wr, 1e6)} | {fmt(spr, 1)} | {fmt(occ, 1, 1)} |\n")
    print(json.dumps(rec))
    return 0


if __name__ == "__main__":
    sys.exit(main())
