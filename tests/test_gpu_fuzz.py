"""Seeded random shapes against the oracle, on every entry point (GPU).

Each case draws its sizes, output type and (for dense calls) an x that starts one element past
a 16-byte boundary from a fixed seed, so every run checks the same cases. Sizes stay small enough
for the oracle to compute every output; the comparison is element by element under the parity
tolerance of test_gpu_parity.py (and the FFN bound of test_gpu_ffn.py).
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

from test_gpu_parity import DEV, assert_parity, assert_swiglu_parity, host
from test_gpu_ffn import assert_ffn_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_state():
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    yield
    assert nv.device_status() == 0


def _k(rng, aligned):
    return int(256 * rng.integers(1, 33)) if aligned else int(16 * rng.integers(1, 257))


def _out(rng):
    return torch.bfloat16 if rng.integers(0, 2) else torch.float32


@pytest.mark.parametrize("case", range(24))
def test_dense_random(case):
    rng = np.random.default_rng(5000 + case)
    N, K, M = int(rng.integers(1, 6001)), _k(rng, case % 3 != 0), int(rng.integers(1, 9))
    p = synth.dense_problem(N, K, M, 5000 + case)
    x = p["x"].to(DEV)
    if case % 5 == 4:  # x one element past a 16-byte boundary
        buf = torch.empty(M * K + 8, dtype=torch.bfloat16, device=DEV)
        x = buf[1:1 + M * K].view(M, K)
        x.copy_(p["x"].to(DEV))
    out = _out(rng)
    y = nv.gemv(p["w"].to(DEV), p["s"].to(DEV), p["g"], x, out_dtype=out)
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, f"dense {N}x{K} M={M} {out}")


@pytest.mark.parametrize("case", range(8))
def test_gate_up_and_swiglu_random(case):
    rng = np.random.default_rng(5100 + case)
    N, K, M = int(rng.integers(1, 4001)), _k(rng, case % 2 == 0), int(rng.integers(1, 9))
    q = synth.gate_up_problem(N, K, M, 5100 + case)
    a = [q[k].to(DEV) if torch.is_tensor(q[k]) else q[k] for k in ("wg", "sg", "gg", "wu", "su", "gu")]
    lim = float(rng.uniform(0.5, 8.0))
    out = _out(rng)
    y = nv.gemv_gate_up(*a, q["x"].to(DEV), out_dtype=out)
    ys = nv.gemv_gate_up_swiglu(*a, q["x"].to(DEV), lim, out_dtype=out)
    torch.cuda.synchronize()
    h = [host(q[k]) if torch.is_tensor(q[k]) else q[k] for k in ("wg", "sg", "gg", "wu", "su", "gu")]
    yr, ya = oracle.gemv_gate_up(*h, synth.bf16_bits(q["x"]))
    assert_parity(y, yr, ya, f"gate_up {N}x{K} M={M}")
    sr, aux = oracle.gate_up_swiglu(*h, synth.bf16_bits(q["x"]), lim)
    assert_swiglu_parity(ys, sr, aux, lim, f"swiglu {N}x{K} M={M} lim={lim:.2f}")


@pytest.mark.parametrize("case", range(10))
def test_moe_random(case):
    rng = np.random.default_rng(5200 + case)
    E = int(rng.choice([8, 64, 288]))
    N, K = 16 * int(rng.integers(1, 129)), _k(rng, case % 4 != 3)
    top_k = int(rng.choice([1, 2, 4, 8]))
    T = int(rng.integers(1, 256 // top_k + 1))
    T = min(T, 32)
    xps = bool(rng.integers(0, 2))
    p = synth.moe_problem(E, N, K, T, top_k, xps, seed=5200 + case)
    out = _out(rng)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv(p["w"].to(DEV), p["s"].to(DEV), p["gs"].to(DEV), p["ids"].to(DEV), p["x"].to(DEV), xps,
                    top_k, out_dtype=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]), synth.bf16_bits(p["x"]),
                                  xps, top_k)
    assert bad == 0
    assert_parity(y, yr, ya, f"moe E={E} {N}x{K} T={T} top{top_k} xps={xps}")


@pytest.mark.parametrize("case", range(6))
def test_sdict_random(case):
    rng = np.random.default_rng(5300 + case)
    N, K, M = int(rng.integers(1, 5001)), _k(rng, True), int(rng.integers(1, 9))
    p = synth.sdict_problem(N, K, M, 5300 + case)
    plane, table = synth.sdict_form(p["s"])
    y = nv.gemv_sdict(p["w"].to(DEV), plane.to(DEV), table.to(DEV), p["g"], p["x"].to(DEV), out_dtype=_out(rng))
    torch.cuda.synchronize()
    yr, ya = oracle.gemv_sdict(host(p["w"]), host(plane), host(table), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, f"sdict {N}x{K} M={M}")


@pytest.mark.parametrize("case", range(8))
def test_ffn_random(case):
    rng = np.random.default_rng(5400 + case)
    H, I, M = 256 * int(rng.integers(1, 17)), 256 * int(rng.integers(1, 13)), int(rng.integers(1, 9))
    p = synth.ffn_problem(H, I, M, 5400 + case)
    lim = float(rng.uniform(0.5, 8.0))
    a = [p[k].to(DEV) if torch.is_tensor(p[k]) else p[k] for k in
         ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    y = nv.ffn_swiglu(*a, p["x"].to(DEV), lim, out_dtype=_out(rng))
    torch.cuda.synchronize()
    hp = [host(p[k]) if torch.is_tensor(p[k]) else p[k] for k in
          ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    yr, ya, aux = oracle.ffn_swiglu(*hp, synth.bf16_bits(p["x"]), lim)
    assert_ffn_parity(y, yr, ya, aux, hp[6], hp[7], hp[8], lim, f"ffn {H}/{I} M={M} "
                      f"{nv.describe_plan('ffn', M, H, I).split()[0]}")
