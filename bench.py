#!/usr/bin/env python
"""Benchmark of the NVFP4 weight-only GEMV hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload W]

A step is one pass of the hot path over one batch of synthetic input. With the default
workload ("vocab"), a step is the vocabulary-head GEMV N x K = 151936 x 4096 at M = 1 with
fp32 output, the largest single-GPU configuration. Every other target step runs in the same
invocation and is reported under "per_workload": the attention projections (4096 x 4096 and
1024 x 4096 at M = 1 and 5, the MUL_MAT shapes of "llama.cpp eval-callback — ggml op level"),
the FFN gate/up + down pair at M = 1, 2, 4, 8, the pair with the fused SwiGLU, and the
288-expert MoE layer at 4 and 32 tokens. Weights are ~N(0, 0.02) quantised to NVFP4, and x is
~N(0, 1) in bf16. Weight copies rotate through a pool larger than twice the L2, so no call
finds its weights in cache.

The timed region is K steps enqueued behind a short torch sleep kernel. The host queues
every launch before the GPU starts, so the measurement is device time. CUDA events
bracket the region and every launch. After each timed region a sample of every call's output
is checked against the CPU oracle; a mismatch marks the line invalid and the exit status is 4.
The script prints one JSON line: the weight-GB/s value, per-call microseconds and roofline
fractions, the dominant kernel's roofline entry, an end-to-end number through the public API
with host buffers, the oracle's CPU baseline and the SM clocks sampled during the region.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMV weight-GB/s and µs/call at M=1..8; % of 8 TB/s HBM roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# (kind, N, K, M, seed, out)   kind: dense | gate_up (N per half) | moe_gate_up | moe_down
SWIGLU_CLAMP = 10.0  # the pages name a clamp in the fused activation but give no limit

WORKLOADS = {
    "attn": ("attention projections N=4096,K=4096 and N=1024,K=4096 at M=1 and M=5, bf16 out",
             [("dense", 4096, 4096, 1, 1, "bf16"), ("dense", 1024, 4096, 1, 3, "bf16"),
              ("dense", 4096, 4096, 5, 2, "bf16"), ("dense", 1024, 4096, 5, 4, "bf16")]),
    "ffn": ("FFN gate+up N=2x12288,K=4096 then down N=4096,K=12288 at M=1, fp32 out",
            [("gate_up", 12288, 4096, 1, 5, "f32"), ("dense", 4096, 12288, 1, 6, "f32")]),
    "ffn_m2": ("FFN gate+up then down at M=2, fp32 out",
               [("gate_up", 12288, 4096, 2, 5, "f32"), ("dense", 4096, 12288, 2, 6, "f32")]),
    "ffn_m4": ("FFN gate+up then down at M=4, fp32 out",
               [("gate_up", 12288, 4096, 4, 5, "f32"), ("dense", 4096, 12288, 4, 6, "f32")]),
    "ffn_m8": ("FFN gate+up then down at M=8, fp32 out",
               [("gate_up", 12288, 4096, 8, 5, "f32"), ("dense", 4096, 12288, 8, 6, "f32")]),
    "ffn_swiglu": ("FFN gate+up N=2x12288,K=4096 with the fused SwiGLU (clamp 10, bf16 [1, 12288] out) "
                   "then down N=4096,K=12288 at M=1 on its own x input, fp32 out",
                   [("gate_up_swiglu", 12288, 4096, 1, 5, "bf16"), ("dense", 4096, 12288, 1, 6, "f32")]),
    "ffn_fused": ("FFN block in one call: gate+up 2x12288x4096 with the SwiGLU (clamp 10) into a bf16 h, "
                  "then down 4096x12288, M=1, fp32 out",
                  [("ffn_block", 4096, 12288, 1, 5, "f32")]),
    "ffn_fused_m2": ("FFN block in one call at M=2, fp32 out", [("ffn_block", 4096, 12288, 2, 5, "f32")]),
    "ffn_shared": ("shared-expert FFN in two calls: gate+up N=2x768,K=4096 with the fused SwiGLU (clamp 10, bf16 "
                   "[2, 768] out), then down N=4096,K=768, M=2, bf16 out",
                   [("gate_up_swiglu", 768, 4096, 2, 9, "bf16"), ("dense", 4096, 768, 2, 10, "bf16")]),
    "ffn_shared_fused": ("shared-expert FFN in one call (gate+up 2x768x4096, SwiGLU, bf16 h, down 4096x768), "
                         "M=2, bf16 out", [("ffn_block", 4096, 768, 2, 9, "bf16")]),
    "card_m2": ("the card's W4A16 calls at decode: KDA in-proj N=8726,K=4096 M=2; KDA o_proj N=4096,K=2816 M=2; "
                "shared gate|up N=768+768,K=4096 M=2; shared down N=4096,K=768 M=2 (bf16 out); routed gate or up, "
                "8 slots of 288 experts, N=704,K=4096 (fp32 out)",
                [("dense", 8726, 4096, 2, 11, "bf16"), ("dense", 4096, 2816, 2, 12, "bf16"),
                 ("gate_up", 768, 4096, 2, 13, "bf16"), ("dense", 4096, 768, 2, 14, "bf16"),
                 ("moe_gate_up", 704, 4096, 1, 15, "f32")]),
    "vocab": ("vocab head N=151936,K=4096,M=1, fp32 out", [("dense", 151936, 4096, 1, 7, "f32")]),
    "moe": ("routed experts: 288 experts, gate_up [3072,4096] then down [4096,1536], "
            "4 tokens x top-8, fp32 per-slot out",
            [("moe_gate_up", 3072, 4096, 4, 8, "f32"), ("moe_down", 4096, 1536, 4, 8, "f32")]),
    "moe_sdict": ("routed experts with dictionary scales (4.3125 bit/weight): 288 experts, gate_up [3072,4096] "
                  "then down [4096,1536], 4 tokens x top-8, fp32 per-slot out",
                  [("moe_sdict_gate_up", 3072, 4096, 4, 8, "f32"), ("moe_sdict_down", 4096, 1536, 4, 8, "f32")]),
    "vocab_sdict": ("vocab head with dictionary scales (4.3125 bit/weight) N=151936,K=4096,M=1, fp32 out",
                    [("dense_sdict", 151936, 4096, 1, 7, "f32")]),
    "moe_t32": ("routed experts at a larger batch: 288 experts, gate_up [3072,4096] then down [4096,1536], "
                "32 tokens x top-8 (256 slots), fp32 per-slot out",
                [("moe_gate_up", 3072, 4096, 32, 8, "f32"), ("moe_down", 4096, 1536, 32, 8, "f32")]),
}


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha256():
    import hashlib
    with open(os.path.join(ROOT, "nvfp4_weight_only_gemv_gb300", "csrc", "nvfp4_gemv.cu"), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_traffic(workload):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or None when
    the summary was taken on another version of the kernel source (or is absent)."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha256") != kernel_source_sha256():
            return None
        return rec.get("dram_bytes_per_launch", {}).get(workload)
    except (OSError, ValueError):
        return None


def run_env(device):
    """What a result was measured on: GPU, SMs, CUDA, torch, the kernel source's hash and the git
    commit when the tree has one."""
    env = {"kernel_source_sha256": kernel_source_sha256()}
    try:
        props = torch.cuda.get_device_properties(device)
        env.update(gpu=props.name, sm_count=props.multi_processor_count,
                   cc=f"{props.major}.{props.minor}", cuda=torch.version.cuda, torch=torch.__version__)
    except Exception:  # no device: the reference arm on a CPU-only host
        env.update(torch=torch.__version__)
    try:
        sha = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True, text=True,
                             timeout=10).stdout.strip()
        env["git_sha"] = sha or None
    except Exception:
        env["git_sha"] = None
    return env


def kernels_of(calls):
    """Names of the library kernels the step's calls launch (from the library's own plan)."""
    import nvfp4_weight_only_gemv_gb300 as nv
    names = {"tile": "gemv_tile_kernel", "tile_moe": "gemv_tile_kernel (MoE)", "stream": "gemv_stream_kernel",
             "tile_sk_moe": "gemv_tile_sk_kernel (MoE)", "tile_swiglu": "gemv_tile_kernel (gate/up + SwiGLU)",
             "stream_moe": "gemv_stream_kernel (MoE)", "simple": "gemv_simple_kernel",
             "tile_sdict": "gemv_tile_kernel (dictionary scales)",
             "tile_sk_moe_sdict": "gemv_tile_sk_kernel (MoE, dictionary scales)",
             "ffn_fused": "gemv_ffn_kernel (gate/up + SwiGLU, readiness counters, down)",
             "ffn_two_launch": "gemv_tile_kernel (gate/up + SwiGLU, then down)"}
    seen = []
    for c in calls:
        if c.kind.startswith("moe"):
            kind = ("moe_per_slot" if c.x_per_slot else "moe") + ("_sdict" if c.sd else "")
            desc = nv.describe_plan(kind, c.E, c.N, c.K, c.T, c.top_k)
        elif c.kind == "ffn_block":
            desc = nv.describe_plan("ffn", c.M, c.N, c.K)
        else:
            kind = c.kind if c.kind in ("gate_up", "gate_up_swiglu", "dense_sdict") else "dense"
            desc = nv.describe_plan(kind, c.M, c.N, c.K)
        name = names.get(desc.split()[0], desc.split()[0])
        if name not in seen:
            seen.append(name)
    return ", ".join(seen) + " (every launch of the step)"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest x over all ranks (a job takes as long as its slowest replica), followed by a
    barrier; x itself when no process group is running."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_gbps(ws: int, bytes_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every replica streams bytes_per_step per step (weak scaling)."""
    return ws * bytes_per_step / (ms_per_step * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the bench runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        try:
            fd, self.path = tempfile.mkstemp(prefix="nvfp4_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except Exception:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if t0 - 0.1 <= r[0] <= t1 + 0.1]
        window = "timed region +-0.1 s"
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
            window = "3 samples nearest the timed region"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ workload construction

class Call:
    """One GEMV of the step, with `copies` independent input sets on the device."""

    def __init__(self, spec, device, copies, gen_device):
        from nvfp4_weight_only_gemv_gb300 import synth
        self.kind, self.N, self.K, self.M, self.seed, out = spec
        self.out_dtype = torch.bfloat16 if out == "bf16" else torch.float32
        self.out_bytes = 2 if out == "bf16" else 4
        self.device = device
        self.sets = []
        self.sd = "sdict" in self.kind    # dictionary scales: s is the index plane, sd its table
        if self.kind == "dense":
            p = synth.dense_problem(self.N, self.K, self.M, self.seed, device=gen_device)
            base = {"w": p["w"], "s": p["s"], "g": p["g"], "x": p["x"]}
            self.rows = self.N
            self.y_shape = (self.M, self.N)
        elif self.kind == "dense_sdict":
            p = synth.sdict_problem(self.N, self.K, self.M, self.seed, device=gen_device)
            plane, table = synth.sdict_form(p["s"])
            base = {"w": p["w"], "s": plane, "sd": table, "g": p["g"], "x": p["x"]}
            self.rows = self.N
            self.y_shape = (self.M, self.N)
        elif self.kind in ("gate_up", "gate_up_swiglu"):
            p = synth.gate_up_problem(self.N, self.K, self.M, self.seed, device=gen_device)
            base = p
            self.rows = 2 * self.N
            self.y_shape = (self.M, self.N if self.kind == "gate_up_swiglu" else 2 * self.N)
        elif self.kind == "ffn_block":
            # N = H (x and y width), K = I (the intermediate width)
            p = synth.ffn_problem(self.N, self.K, self.M, self.seed, device=gen_device)
            base = {k: v for k, v in p.items() if k not in ("H", "I", "M")}
            self.rows = self.N
            self.y_shape = (self.M, self.N)
        else:
            self.T, self.top_k, self.E = self.M, 8, 288
            self.x_per_slot = self.kind.endswith("_down")
            p = synth.moe_problem(self.E, self.N, self.K, self.T, self.top_k, self.x_per_slot,
                                  seed=self.seed, device=gen_device,
                                  fill="all" if copies > 1 else "routed", max_codes=32 if self.sd else None)
            base = dict(p)
            if self.sd:
                base["s"], base["sd"] = synth.sdict_form(p["s"])
            self.rows = self.N
            self.y_shape = (self.T * self.top_k, self.N)
        self.host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in base.items()}
        for c in range(copies):
            d = {}
            for k, v in base.items():
                if isinstance(v, torch.Tensor):
                    if self.kind.startswith("moe") and k in ("w", "s", "sd") and c > 0:
                        d[k] = self.sets[0][k]          # expert tensors are already > 2x L2
                    else:
                        d[k] = v.to(device).clone()
                else:
                    d[k] = v
            if self.kind.startswith("moe") and c > 0:
                d["ids"] = synth.routing(self.T, self.top_k, self.E, self.seed * 7919 + c).to(device)
            d["y"] = torch.empty(self.y_shape, dtype=self.out_dtype, device=device)
            if self.kind == "ffn_block":
                import nvfp4_weight_only_gemv_gb300 as nv
                d["ws"] = nv.ffn_workspace(self.M, self.K, device)
            self.sets.append(d)

    # bytes -------------------------------------------------------------
    def unique_experts(self, c):
        if not hasattr(self, "_uniq"):
            self._uniq = {}
        if c not in self._uniq:
            self._uniq[c] = len(set(self.sets[c]["ids"].tolist()))
        return self._uniq[c]

    def weight_bytes(self, c=0):
        # dictionary scales: a 5-bit index per 16 weights (plus a 32-byte table per tensor)
        per_row = self.K * 0.5 + (self.K * 5 / 128 if self.sd else self.K / 16)
        if self.kind in ("gate_up", "gate_up_swiglu"):
            return 2 * self.N * per_row
        if self.kind == "ffn_block":
            return 3 * self.N * per_row  # gate and up [I, H], down [H, I]: 3 * H * I weights
        if self.kind.startswith("moe"):
            return self.unique_experts(c) * (self.N * per_row + (32 if self.sd else 0))
        return self.N * per_row + (32 if self.sd else 0)

    def alg_bytes(self, c=0):
        """Bytes of the roofline formula: weights + x + y."""
        if self.kind.startswith("moe"):
            slots = self.T * self.top_k
            xrows = slots if self.x_per_slot else self.T
            return self.weight_bytes(c) + xrows * self.K * 2 + slots * self.N * self.out_bytes
        if self.kind == "ffn_block":  # x [M, H] in, y [M, H] out; h stays inside the call
            return self.weight_bytes(c) + self.M * self.N * (2 + self.out_bytes)
        return self.weight_bytes(c) + self.M * self.K * 2 + self.M * self.y_shape[1] * self.out_bytes

    def x_bytes(self):
        return self.sets[0]["x"].numel() * 2

    def y_bytes(self):
        return self.sets[0]["y"].numel() * self.out_bytes

    # launches ----------------------------------------------------------
    def launch(self, c, x=None, y=None):
        import nvfp4_weight_only_gemv_gb300 as nv
        d = self.sets[c]
        x = d["x"] if x is None else x
        y = d["y"] if y is None else y
        if self.kind == "dense":
            nv.gemv(d["w"], d["s"], d["g"], x, out=y)
        elif self.kind == "dense_sdict":
            nv.gemv_sdict(d["w"], d["s"], d["sd"], d["g"], x, out=y)
        elif self.sd:
            nv.moe_gemv_sdict(d["w"], d["s"], d["sd"], d["gs"], d["ids"], x, self.x_per_slot, self.top_k, out=y)
        elif self.kind == "gate_up":
            nv.gemv_gate_up(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], x, out=y)
        elif self.kind == "gate_up_swiglu":
            nv.gemv_gate_up_swiglu(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], x, SWIGLU_CLAMP, out=y)
        elif self.kind == "ffn_block":
            nv.ffn_swiglu(d["wg"], d["sg"], d["gg"], d["wu"], d["su"], d["gu"], d["wd"], d["sd"], d["gd"], x,
                          SWIGLU_CLAMP, workspace=d["ws"], out=y)
        else:
            nv.moe_gemv(d["w"], d["s"], d["gs"], d["ids"], x, self.x_per_slot, self.top_k, out=y)
        return y

    # oracle ------------------------------------------------------------
    def oracle_rows(self, frac, rng):
        cols = self.y_shape[1] if self.kind == "gate_up_swiglu" else self.rows  # output columns
        n = max(1, int(round(cols * frac)))
        return np.sort(rng.choice(cols, size=min(n, cols), replace=False)).astype(np.int64)

    def run_oracle(self, rows):
        import oracle
        from nvfp4_weight_only_gemv_gb300 import synth
        h = self.host
        if self.kind == "dense":
            oracle.gemv(h["w"].numpy(), h["s"].numpy(), h["g"], synth.bf16_bits(h["x"]), rows=rows)
            return len(rows) * (self.K * 0.5 + self.K / 16)
        if self.kind == "dense_sdict":
            oracle.gemv_sdict(h["w"].numpy(), h["s"].numpy(), h["sd"].numpy(), h["g"], synth.bf16_bits(h["x"]),
                              rows=rows)
            return len(rows) * (self.K * 0.5 + self.K * 5 / 128)
        if self.kind == "gate_up":
            oracle.gemv_gate_up(h["wg"].numpy(), h["sg"].numpy(), h["gg"], h["wu"].numpy(), h["su"].numpy(),
                                h["gu"], synth.bf16_bits(h["x"]), rows=rows)
            return len(rows) * (self.K * 0.5 + self.K / 16)
        if self.kind == "gate_up_swiglu":
            oracle.gate_up_swiglu(h["wg"].numpy(), h["sg"].numpy(), h["gg"], h["wu"].numpy(), h["su"].numpy(),
                                  h["gu"], synth.bf16_bits(h["x"]), SWIGLU_CLAMP, rows=rows)
            return 2 * len(rows) * (self.K * 0.5 + self.K / 16)  # a gate and an up row per output
        if self.kind == "ffn_block":
            oracle.ffn_swiglu(*ffn_host_args(h), synth.bf16_bits(h["x"]), SWIGLU_CLAMP, rows=rows)
            # every gate and up row (h is needed whole), and the sampled down rows
            return (2 * self.K + len(rows)) * (self.N * 0.5 + self.N / 16)
        ids = self.sets[0]["ids"].cpu().numpy()
        if self.sd:
            oracle.moe_gemv_sdict(h["w"].numpy(), h["s"].numpy(), h["sd"].numpy(), h["gs"].numpy(), ids,
                                  synth.bf16_bits(h["x"]), self.x_per_slot, self.top_k, rows=rows)
        else:
            oracle.moe_gemv(h["w"].numpy(), h["s"].numpy(), h["gs"].numpy(), ids, synth.bf16_bits(h["x"]),
                            self.x_per_slot, self.top_k, rows=rows)
        # the oracle walks every slot; count the bytes of the slots it read
        return len(ids) * len(rows) * (self.K * 0.5 + (self.K * 5 / 128 if self.sd else self.K / 16))


def pool_copies(calls_spec, device):
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    per_step, moe = 0, False
    for kind, N, K, M, *_ in calls_spec:
        rows = {"gate_up": 2 * N, "gate_up_swiglu": 2 * N, "ffn_block": 3 * N}.get(kind, N)
        if kind.startswith("moe"):
            moe = True
        else:
            per_step += rows * K * 9 // 16
    notes = []
    copies = 4 if moe else 1
    if per_step:
        copies = max(copies, math.ceil(2.5 * l2 / per_step))
        notes.append(f"{copies} rotating weight copies ({copies * per_step / 1e6:.0f} MB > 2x L2 of {l2 / 1e6:.0f} MB)")
    if moe:
        notes.append(f"routing rotates over {copies} id sets; the expert tensors (all experts, counted by the "
                     "distinct experts a step reads) exceed 2x L2")
    return copies, l2, "; ".join(notes)


# ------------------------------------------------------------------ timing

def timed_region(calls, copies, steps, gate_cycles, stream):
    """The timed region: `steps` steps enqueued back to back behind a sleep kernel, with CUDA
    events only at its two ends, so consecutive GEMVs can overlap as they would in a decode
    step. Returns (region_ms, host_s, gate_ms)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    e_gate, e_start, e_end = ev(), ev(), ev()
    e_gate.record(stream)
    torch.cuda._sleep(int(gate_cycles))
    e_start.record(stream)
    h0 = time.perf_counter()
    for st in range(steps):
        c = st % copies
        for call in calls:
            call.launch(c)
    e_end.record(stream)
    host_s = time.perf_counter() - h0
    e_end.synchronize()
    return e_start.elapsed_time(e_end), host_s, e_gate.elapsed_time(e_start)


def per_call_region(calls, copies, steps, gate_cycles, stream):
    """Diagnostic pass: an event pair around every launch (isolated per-call times)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    pairs = [[(ev(), ev()) for _ in range(steps)] for _ in calls]
    torch.cuda._sleep(int(gate_cycles))
    for st in range(steps):
        c = st % copies
        for ci, call in enumerate(calls):
            a, b = pairs[ci][st]
            a.record(stream)
            call.launch(c)
            b.record(stream)
    torch.cuda.synchronize()
    return [[a.elapsed_time(b) for a, b in pairs[ci]] for ci in range(len(calls))]


def e2e_region(calls, copies, steps, stream, device, graph=False):
    """Public API end to end: pinned host x -> device, the step's GEMVs, y -> pinned host, and
    a synchronize, every step. graph=True captures each rotation copy's step (copies, calls
    and all) in a CUDA graph once, outside the timed region, and replays one graph per step,
    the way a decode loop drives the library; eager mode issues every call from Python."""
    hx = [[c.sets[k]["x"].cpu().pin_memory() for k in range(copies)] for c in calls]
    hy = [torch.empty(c.y_shape, dtype=c.out_dtype).pin_memory() for c in calls]
    dx = [torch.empty_like(c.sets[0]["x"]) for c in calls]

    def step(k):
        for ci, c in enumerate(calls):
            dx[ci].copy_(hx[ci][k], non_blocking=True)
            y = c.launch(k, x=dx[ci])
            hy[ci].copy_(y, non_blocking=True)

    graphs = None
    if graph:
        side = torch.cuda.Stream(device=device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):  # warm the library's per-kernel setup outside capture
            step(0)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graphs = []
        for k in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(k)
            graphs.append(g)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for st in range(steps):
        k = st % copies
        if graphs is not None:
            graphs[k].replay()
            torch.cuda.current_stream().synchronize()
        else:
            step(k)
            stream.synchronize()
    t1 = time.perf_counter()
    return (t1 - t0) * 1e3 / steps


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_pass(calls, target_s):
    """The oracle over a row sample of every GEMV of the step, the sample grown until one timed
    pass takes about target_s / 3; once every row is in the sample, whole steps are repeated.
    Returns (bytes, seconds, sample description)."""
    rng = np.random.default_rng(0)
    frac, reps = 0.002, 1
    t = 0.0
    byts = 0.0
    for _ in range(4):
        t0 = time.perf_counter()
        byts = sum(c.run_oracle(c.oracle_rows(frac, rng)) for _ in range(reps) for c in calls)
        t = time.perf_counter() - t0
        if t > target_s / 3:
            break
        grow = max(2.0, target_s / max(t, 1e-3))
        if frac < 1.0:
            frac = min(1.0, frac * grow)
        else:
            reps = int(math.ceil(reps * grow))
    what = f"{frac * 100:.3g}% of the output rows of every GEMV of one step"
    if reps > 1:
        what = f"every GEMV of one step, {reps} times"
    return byts, t, f"{what} ({byts / 1e6:.1f} MB of weights, {t:.2f} s wall)"


def cpu_baseline(calls, target_s=6.0, single_thread=True):
    """The oracle on the host cores over a bounded sample of the step (all OpenMP threads), and
    the same on one thread when single_thread is set."""
    import oracle
    byts, t, sample = _oracle_pass(calls, target_s)
    res = {"value": byts / t / 1e9, "unit": "GB/s (NVFP4 weight bytes)", "cores": oracle.threads(),
           "kind": "oracle", "sample": sample, "cpu": cpu_model()}
    if single_thread:
        n = oracle.threads()
        oracle.set_threads(1)
        try:
            b1, t1, sample1 = _oracle_pass(calls, target_s / 3)
        finally:
            oracle.set_threads(n)
        res["one_thread"] = {"value": b1 / t1 / 1e9, "cores": 1, "sample": sample1}
    return res


# ------------------------------------------------------------------ in-run parity

def ffn_host_args(h):
    return [h[k].numpy() if isinstance(h[k], torch.Tensor) else h[k] for k in
            ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]


def _swiglu_bound(aux, y_ref, lim):
    """The fused activation's bound: the GEMV bound of gate and up carried through the clamp and
    silu (|silu'| <= 1.1, |silu(v)| <= max(|v|, 0.28)), plus the fp32 evaluation."""
    tg, tu = 1e-5 * aux["gate_abs"] + 1e-6, 1e-5 * aux["up_abs"] + 1e-6
    cg = np.clip(aux["gate"], -lim, lim)
    cu = np.clip(aux["up"], -lim, lim)
    return (1.1 * np.abs(cu) * tg + np.maximum(np.abs(cg), 0.28) * tu + 1.1 * tg * tu
            + 1e-6 * np.abs(np.nan_to_num(y_ref)) + 1e-6)


def _ffn_flip_bound(h, aux, rows, lim):
    """The FFN's extra term: where a bf16 rounding boundary lies within the activation's bound of
    the oracle's h, the GPU's bf16 h may differ by that bound plus two bf16 steps; the down
    GEMV's A-scale on those differences (oracle only) bounds what they move y."""
    import oracle
    hh, hb = aux["h"], aux["h_bits"]
    e = _swiglu_bound(aux, hh, lim)
    mb = (hb & 0x7FFF).astype(np.int64)
    val = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    hv = val(mb.astype(np.uint16))
    lo = np.where(mb > 0, val(np.maximum(mb - 1, 0).astype(np.uint16)), -2.0 ** -133)
    hi = val(np.minimum(mb + 1, 0x7F80).astype(np.uint16))
    a = np.abs(hh)
    near = ((a - (lo + hv) / 2 <= e) | ((hv + hi) / 2 - a <= e)) & np.isfinite(hh)
    d = np.where(near, e + 2 * np.maximum(hv - lo, hi - hv), 0.0)
    _, bound = oracle.gemv(h["wd"].numpy(), h["sd"].numpy(), h["gd"], oracle.bf16_rne(d * (1 + 2.0 ** -7)), rows=rows)
    return np.nan_to_num(bound)


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -126)
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def check_outputs(calls, n_cols=48, seed=5):
    """The timed outputs against the oracle: for every call, copy 0's output (written inside the
    timed region) on a sample of n_cols output columns, compared with the oracle's value of
    those columns on the same inputs, under the parity tolerance |y - y_ref| <= 1e-5 * A + 1e-6
    (A = |g| * sum_k |w_k x_k|), plus one bf16 ulp of y_ref for bf16 output; the fused SwiGLU
    carries that bound through the activation. NaN must match NaN. Returns a summary dict."""
    import oracle
    from nvfp4_weight_only_gemv_gb300 import synth
    rng = np.random.default_rng(seed)
    checked, bad = 0, 0
    worst = 0.0
    for c in calls:
        h = c.host
        cols = c.y_shape[1]
        rows = np.sort(rng.choice(cols, size=min(n_cols, cols), replace=False)).astype(np.int64)
        y = c.sets[0]["y"].float().cpu().numpy().astype(np.float64)[:, rows]
        bf = c.out_dtype == torch.bfloat16
        if c.kind == "dense":
            yr, ya = oracle.gemv(h["w"].numpy(), h["s"].numpy(), h["g"], synth.bf16_bits(h["x"]), rows=rows)
            tol = 1e-5 * ya + 1e-6
        elif c.kind == "dense_sdict":
            yr, ya = oracle.gemv_sdict(h["w"].numpy(), h["s"].numpy(), h["sd"].numpy(), h["g"],
                                       synth.bf16_bits(h["x"]), rows=rows)
            tol = 1e-5 * ya + 1e-6
        elif c.kind == "gate_up":
            yr, ya = oracle.gemv_gate_up(h["wg"].numpy(), h["sg"].numpy(), h["gg"], h["wu"].numpy(),
                                         h["su"].numpy(), h["gu"], synth.bf16_bits(h["x"]), rows=rows)
            tol = 1e-5 * ya + 1e-6
        elif c.kind == "gate_up_swiglu":
            yr, aux = oracle.gate_up_swiglu(h["wg"].numpy(), h["sg"].numpy(), h["gg"], h["wu"].numpy(),
                                            h["su"].numpy(), h["gu"], synth.bf16_bits(h["x"]), SWIGLU_CLAMP,
                                            rows=rows)
            tol = _swiglu_bound(aux, yr, SWIGLU_CLAMP)
        elif c.kind == "ffn_block":
            yr, ya, aux = oracle.ffn_swiglu(*ffn_host_args(h), synth.bf16_bits(h["x"]), SWIGLU_CLAMP, rows=rows)
            tol = 1e-5 * ya + 1e-6 + _ffn_flip_bound(h, aux, rows, SWIGLU_CLAMP)
        else:
            ids = c.sets[0]["ids"].cpu().numpy()
            if c.sd:
                yr, ya, _ = oracle.moe_gemv_sdict(h["w"].numpy(), h["s"].numpy(), h["sd"].numpy(), h["gs"].numpy(),
                                                  ids, synth.bf16_bits(h["x"]), c.x_per_slot, c.top_k, rows=rows)
            else:
                yr, ya, _ = oracle.moe_gemv(h["w"].numpy(), h["s"].numpy(), h["gs"].numpy(), ids,
                                            synth.bf16_bits(h["x"]), c.x_per_slot, c.top_k, rows=rows)
            tol = 1e-5 * ya + 1e-6
        if bf:
            tol = tol + _ulp_bf16(np.nan_to_num(yr))
        nan_r = np.isnan(yr)
        err = np.where(nan_r, 0.0, np.abs(y - yr))
        miss = (np.isnan(y) != nan_r) | (err > tol)
        bad += int(miss.sum())
        checked += y.size
        worst = max(worst, float(np.max(np.where(nan_r, 0.0, err / tol))) if y.size else 0.0)
    return {"ok": bad == 0, "checked": checked, "outside_tolerance": bad, "worst_err_over_tol": round(worst, 4),
            "method": f"oracle on {n_cols} sampled output columns of every call (copy 0, written in the "
                      "timed region), parity tolerance"}


# ------------------------------------------------------------------ arms

def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on a bounded row sample per step."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    desc, spec = WORKLOADS[args.workload]
    device = "cpu"
    calls = [Call(s, device, 1, "cpu") for s in spec]
    rng = np.random.default_rng(1)
    # size the per-step sample so that warmup + steps take about a minute
    frac = 0.002
    t0 = time.perf_counter()
    for c in calls:
        c.run_oracle(c.oracle_rows(frac, rng))
    t_probe = max(time.perf_counter() - t0, 1e-4)
    frac = min(1.0, frac * (60.0 / (args.steps + args.warmup)) / t_probe)
    for _ in range(args.warmup):
        for c in calls:
            c.run_oracle(c.oracle_rows(frac, rng))
    tot_t, tot_b = 0.0, 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        b = sum(c.run_oracle(c.oracle_rows(frac, rng)) for c in calls)
        tot_t += time.perf_counter() - t0
        tot_b += b
    value = tot_b / tot_t / 1e9
    sample = f"{frac * 100:.3g}% of the output rows of every GEMV per step"
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "GB/s (NVFP4 weight bytes)",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {desc}"},
            "cpu_baseline": {"value": value, "unit": "GB/s (NVFP4 weight bytes)", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s (NVFP4 weight bytes)", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "env": run_env(None)}
    print(json.dumps(line))
    return 0


PER_WORKLOAD = ["attn", "card_m2", "ffn", "ffn_m2", "ffn_m4", "ffn_m8", "ffn_swiglu", "ffn_fused", "ffn_shared",
                "ffn_shared_fused", "moe", "moe_t32", "moe_sdict", "vocab_sdict"]


def measure(name, steps, warmup, device, stream, ws, sampler=None):
    """One workload: build its calls, warm up, time `steps` steps back to back, time every call
    in isolation, check sampled outputs against the oracle. Returns (calls, copies, record)."""
    desc, spec = WORKLOADS[name]
    copies, l2, l2_note = pool_copies(spec, device)
    calls = [Call(s, device, copies, "cuda") for s in spec]

    # warm-up (also measures the host enqueue rate to size the gate)
    h0 = time.perf_counter()
    for st in range(max(3, warmup)):
        for c in calls:
            c.launch(st % copies)
    torch.cuda.synchronize()
    per_launch_host = (time.perf_counter() - h0) / (max(3, warmup) * len(calls))
    sm_mhz_guess = 1900.0
    gate_ms = max(5.0, 3.0 * per_launch_host * 1e3 * steps * len(calls) + 2.0)

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    region_ms, host_s, gate_meas = timed_region(calls, copies, steps, gate_ms * 1e3 * sm_mhz_guess, stream)
    if host_s * 1e3 > gate_meas:   # host could not stay ahead: retry once with a longer gate
        gate_ms = host_s * 1e3 * 3 + 5
        region_ms, host_s, gate_meas = timed_region(calls, copies, steps, gate_ms * 1e3 * sm_mhz_guess, stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    region_ms = max_over_ranks(region_ms, device)
    parity = check_outputs(calls)
    per_call = per_call_region(calls, copies, min(steps, 100), gate_ms * 2e3 * sm_mhz_guess, stream)

    ms_per_step = region_ms / steps
    wbytes_step = sum(np.mean([c.weight_bytes(k % copies) for k in range(min(copies, steps))]) for c in calls)
    value = job_gbps(ws, wbytes_step, ms_per_step)

    peak, peak_kind = measured_peaks()
    call_rows = []
    step_alg = 0.0
    for ci, c in enumerate(calls):
        ms = float(np.mean(per_call[ci]))
        alg = float(np.mean([c.alg_bytes(k % copies) for k in range(steps)]))
        wb = float(np.mean([c.weight_bytes(k % copies) for k in range(steps)]))
        step_alg += alg
        call_rows.append({"call": c.kind, "N": c.N, "K": c.K, "M": c.M, "out": str(c.out_dtype).split(".")[-1],
                          "us_isolated": round(ms * 1e3, 3),
                          "us_isolated_median": round(float(np.median(per_call[ci])) * 1e3, 3),
                          "weight_GBps_isolated": round(wb / (ms * 1e-3) / 1e9, 1),
                          "alg_bytes": int(alg),
                          "pct_of_8TBps_isolated": round(100 * alg / (ms * 1e-3) / (NOMINAL_HBM_GBS * 1e9), 2)})
    launches = steps * len(calls)
    us_per_launch = region_ms * 1e3 / launches
    achieved = step_alg * steps / (region_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": kernel_traffic(name),
                "kernel": kernels_of(calls),
                "us_per_launch": round(us_per_launch, 3),
                "pct_of_8TBps": round(100 * achieved / NOMINAL_HBM_GBS, 2),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs: copy bandwidth)"}
    rec = {"workload": f"{name}: {desc}", "value": round(value, 2), "ms_per_step": round(ms_per_step, 6),
           "steps": steps, "launches": launches, "l2": l2_note, "calls_per_step": len(calls),
           "calls": call_rows, "roofline": roofline, "parity": parity,
           "wall": (t_wall0, t_wall1),
           "timing": {"gate_ms": round(gate_meas, 3), "host_enqueue_ms": round(host_s * 1e3, 3),
                      "method": "timed region: steps back to back behind a sleep kernel, events at "
                                "both ends; calls[].us_isolated: separate pass, events around "
                                f"each launch ({len(per_call[0])} per call)"}}
    return calls, copies, wbytes_step, rec


def release(calls):
    for c in calls:
        c.sets.clear()
        c.host.clear()
    calls.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_ours(args):
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import nvfp4_weight_only_gemv_gb300 as nv
    nv.library()
    stream = torch.cuda.current_stream(device)
    sampler = ClockSampler(local) if rank == 0 else None

    calls, copies, wbytes_step, rec = measure(args.workload, args.steps, args.warmup, device, stream, ws)
    t_wall0, t_wall1 = rec.pop("wall")
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if sampler:
        sampler.stop()

    e2e_eager_ms = e2e_region(calls, copies, max(args.steps, 10), stream, device)
    try:
        e2e_ms = e2e_region(calls, copies, max(args.steps, 10), stream, device, graph=True)
        e2e_method = ("CUDA graph per step (H2D of x from pinned host memory, the step's GEMVs "
                      "through the public API, D2H of y), replayed and synchronised every step")
    except Exception as exc:  # capture unavailable: report the eager loop alone
        e2e_ms, e2e_method = e2e_eager_ms, f"eager Python loop (graph capture failed: {exc})"
    e2e_ms = max_over_ranks(e2e_ms, device)
    e2e_eager_ms = max_over_ranks(e2e_eager_ms, device)
    e2e = {"value": round(job_gbps(ws, wbytes_step, e2e_ms), 2), "unit": "GB/s (NVFP4 weight bytes)",
           "ms_per_step": round(e2e_ms, 4),
           "h2d_bytes_per_step": int(sum(c.x_bytes() for c in calls)),
           "d2h_bytes_per_step": int(sum(c.y_bytes() for c in calls)),
           "method": e2e_method,
           "eager": {"value": round(job_gbps(ws, wbytes_step, e2e_eager_ms), 2),
                     "ms_per_step": round(e2e_eager_ms, 4),
                     "method": "every copy and call issued from Python each step, then a synchronize"}}

    cpu_on = rank == 0 and ws == 1 and not args.no_cpu_baseline
    base = cpu_baseline(calls) if cpu_on else None
    release(calls)

    # every other target step of the same run, each with its own timed region, oracle check
    # and CPU baseline
    per = {}
    if not args.no_per_workload:
        for name in PER_WORKLOAD:
            if name == args.workload:
                continue
            pc, _, _, prec = measure(name, min(args.steps, 100), args.warmup, device, stream, ws)
            prec.pop("wall")
            if cpu_on:
                b = cpu_baseline(pc, target_s=1.5, single_thread=False)
                prec["cpu_baseline"] = {k: b[k] for k in ("value", "unit", "cores", "sample")}
            release(pc)
            per[name] = prec

    ok = rec["parity"]["ok"] and all(r["parity"]["ok"] for r in per.values())
    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": "GB/s (NVFP4 weight bytes)",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": rec["workload"], "parallelism": f"replicas x{ws}",
                           "l2": rec["l2"], "calls_per_step": rec["calls_per_step"]},
                "calls": rec["calls"], "roofline": rec["roofline"], "parity": rec["parity"],
                "cpu_baseline": base, "e2e": e2e,
                "gpu_launches": rec["launches"], "clocks": clocks, "env": run_env(device),
                "timing": rec["timing"],
                "per_workload": {k: {"workload": v["workload"], "value": v["value"],
                                     "ms_per_step": v["ms_per_step"], "steps": v["steps"],
                                     "frac": v["roofline"]["frac"], "us_per_launch": v["roofline"]["us_per_launch"],
                                     "pct_of_8TBps": v["roofline"]["pct_of_8TBps"],
                                     "traffic": v["roofline"]["traffic"], "kernel": v["roofline"]["kernel"],
                                     "calls": v["calls"], "parity": v["parity"],
                                     "cpu_baseline": v.get("cpu_baseline")} for k, v in per.items()}}
        if not ok:
            line["invalid"] = "a timed output is outside the oracle's tolerance (see parity)"
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0 if ok else 4


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="vocab")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --workload (default: also every other target step, as per_workload)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if argv is None:  # run as a program: a step that never finished must not hold the GPU
        limit = 900 + 2 * (args.steps + args.warmup)
        import threading

        def _expire():
            print(f"bench.py: no result after {limit} s; exiting", file=sys.stderr, flush=True)
            os._exit(3)

        timer = threading.Timer(limit, _expire)
        timer.daemon = True
        timer.start()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
