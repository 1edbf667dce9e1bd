"""GPU parity of the FFN block (nvfp4_ffn_swiglu) against the oracle's FFN.

The FFN is the shared-expert group of "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json" (block
l3.moe: shared_gate_up, shared_clamp, shared_act, shared_down): h = bf16(silu(c(gate)) * c(up)),
then y = g_down * W_down . h. Shapes: the 12288-wide FFN of "llama.cpp eval-callback — ggml op
level" (ffn_gate/ffn_up [4096 -> 12288], ffn_down [12288 -> 4096]), the routed-expert widths of
the card (4096 x 1536), small and ragged cases. Inputs come from the seeded generator only.

Tolerance (derived in the design notes, reading 19): the GPU's fp32 h differs from the oracle's
fp64 h by at most e_k (the SwiGLU bound); where no bf16 rounding boundary lies within e_k of
h_k both round alike, elsewhere they may differ by d_k = e_k + two bf16 steps. So
    |y - y_ref| <= 1e-5 * A + 1e-6 + |g_down| * sum_k |W_down[n, k]| * d_k  (+ one bf16 ulp),
the last term being the oracle's A-scale of the down GEMV on d, formed from oracle values only.
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

from test_gpu_parity import DEV, host, swiglu_tolerance, assert_swiglu_parity, ulp_bf16

pytestmark = pytest.mark.gpu

HEADER = 2048  # workspace bytes before h: the readiness counters' lines


@pytest.fixture(autouse=True)
def _clean_state():
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    yield
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    assert nv.device_status() == 0


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def flip_allowance(aux, lim):
    """d_k: 0 where the GPU's bf16 h must equal the oracle's, else e_k + two bf16 steps."""
    h, hb = aux["h"], aux["h_bits"]
    e = swiglu_tolerance(aux, h, lim, False)
    mag_bits = (hb & 0x7FFF).astype(np.int64)
    hv = _bf16_values(mag_bits.astype(np.uint16))
    lo = np.where(mag_bits > 0, _bf16_values(np.maximum(mag_bits - 1, 0).astype(np.uint16)), -2.0 ** -133)
    hi = _bf16_values(np.minimum(mag_bits + 1, 0x7F80).astype(np.uint16))
    a = np.abs(h)
    near = (a - (lo + hv) / 2 <= e) | ((hv + hi) / 2 - a <= e)
    step = np.maximum(hv - lo, hi - hv)
    return np.where(near & np.isfinite(h), e + 2 * step, 0.0)


def assert_ffn_parity(y_gpu, y_ref, ya, aux, wd, sd, gd, lim, what=""):
    d = flip_allowance(aux, lim)
    d_bits = oracle.bf16_rne(d * (1 + 2.0 ** -7))  # bf16 at or above d
    _, bound = oracle.gemv(wd, sd, gd, d_bits)
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert y.shape == y_ref.shape
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan_ref), f"{what}: NaN positions differ"
    tol = 1e-5 * ya + 1e-6 + np.nan_to_num(bound)
    if y_gpu.dtype == torch.bfloat16:
        tol = tol + ulp_bf16(np.nan_to_num(y_ref))
    err = np.where(nan_ref, 0.0, np.abs(y - y_ref))
    bad = err > np.where(nan_ref, 1.0, tol)
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={y[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")
    return int((d > 0).sum())


def problem(H, I, M, seed, device="cpu"):
    return synth.ffn_problem(H, I, M, seed, device=device)


def run(p, lim, out_dtype=torch.float32, ws=None):
    args = [p[k].to(DEV) if torch.is_tensor(p[k]) else p[k] for k in
            ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    x = p["x"].to(DEV)
    if ws is None:
        ws = nv.ffn_workspace(p["M"], p["I"])
    y = nv.ffn_swiglu(*args, x, lim, workspace=ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, ws


def reference(p, lim):
    hp = [host(p[k]) if torch.is_tensor(p[k]) else p[k] for k in
          ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    return oracle.ffn_swiglu(*hp, synth.bf16_bits(p["x"]), lim)


def check(p, lim, out_dtype=torch.float32, what=""):
    y, ws = run(p, lim, out_dtype)
    yr, ya, aux = reference(p, lim)
    M, I = p["M"], p["I"]
    h_gpu = ws[HEADER:HEADER + M * I * 2].view(torch.bfloat16).view(M, I)
    assert_swiglu_parity(h_gpu, aux["h"], aux, lim, f"{what} h")
    assert_ffn_parity(y, yr, ya, aux, host(p["wd"]), host(p["sd"]), p["gd"], lim, what)
    assert not torch.any(ws[:HEADER]), "counters left non-zero"
    return y, ws


@pytest.mark.parametrize("M,lim,out", [(1, 10.0, torch.bfloat16), (1, 1.0, torch.float32), (2, 10.0, torch.bfloat16),
                                       (2, 0.5, torch.float32), (4, 2.0, torch.bfloat16)])
def test_ffn_shared_expert_fused(M, lim, out):
    # the graph's shared-expert group: gate|up 768+768 x 4096, down 4096 x 768 (the card's M = 2)
    assert nv.describe_plan("ffn", M, 4096, 768).startswith("ffn_fused ")
    p = problem(4096, 768, M, 800 + M + int(lim * 4), device=DEV)
    check(p, lim, out, f"ffn 4096/768 M={M} lim={lim}")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_ffn_12288_two_launches(M):
    assert nv.describe_plan("ffn", M, 4096, 12288).startswith("ffn_two_launch ")
    p = problem(4096, 12288, M, 810 + M, device=DEV)
    check(p, 10.0, torch.float32, f"ffn 4096/12288 M={M}")


@pytest.mark.parametrize("H,I,M", [(4096, 1536, 1), (4096, 1536, 2), (4096, 1536, 5), (1024, 512, 1),
                                   (1024, 512, 3), (1024, 512, 8), (256, 256, 1), (2048, 768, 4),
                                   (768, 3072, 2), (4096, 4096, 1)])
def test_ffn_small_shapes(H, I, M):
    p = problem(H, I, M, 820 + H % 97 + I % 89 + M)
    check(p, 1.5, torch.float32 if M % 2 else torch.bfloat16, f"ffn {H}/{I} M={M}")


@pytest.mark.parametrize("H,I,M", [(784, 512, 2), (1024, 400, 3), (16, 16, 1), (272, 48, 5)])
def test_ffn_ragged_sizes(H, I, M):
    assert nv.describe_plan("ffn", M, H, I).startswith("ffn_two_launch ")
    p = problem(H, I, M, 830 + H + I + M)
    check(p, 2.0, torch.float32, f"ffn {H}/{I} M={M}")


def test_ffn_fused_plans_cover_the_small_shapes():
    fused = [nv.describe_plan("ffn", M, H, I).split()[0] for H, I, M in
             ((1024, 512, 1), (1024, 512, 3), (1024, 512, 8), (4096, 1536, 1))]
    assert fused.count("ffn_fused") == 4, fused


def test_ffn_repeated_calls_share_a_workspace():
    ws = None
    base = problem(1024, 512, 2, 840)
    for i in range(5):
        p = dict(base, x=synth.random_x(2, 1024, 841 + i))
        y, ws = run(p, 1.0, ws=ws)
        yr, ya, aux = reference(p, 1.0)
        assert_ffn_parity(y, yr, ya, aux, host(p["wd"]), host(p["sd"]), p["gd"], 1.0, f"call {i}")
        assert not torch.any(ws[:HEADER])


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_ffn_other_kernels(variant):
    # 1: byte-load kernels (two launches), 2: the fused kernel in exact fp32 (h read through L2
    # on every box), 3: no tile kernels (two launches)
    nv.set_variant(variant)
    for H, I, M in ((1024, 512, 1), (4096, 1536, 3)):
        p = problem(H, I, M, 850 + variant + M)
        check(p, 1.0, torch.float32, f"ffn variant {variant} {H}/{I} M={M}")


def test_ffn_nan_in_h_poisons_every_output():
    p = problem(1024, 512, 1, 860)
    sg = p["sg"].clone()
    sg[37, 3] = 0x7F  # a NaN scale in gate row 37: h[37] is NaN, and every down row reads it
    p["sg"] = sg
    y, _ = run(p, 1.0)
    yr, ya, aux = reference(p, 1.0)
    assert np.isnan(aux["h"][0, 37]) and np.isnan(yr).all()
    assert torch.isnan(y).all()


def test_ffn_cuda_graph_replay():
    p = problem(1024, 512, 1, 870)
    args = [p[k].to(DEV) if torch.is_tensor(p[k]) else p[k] for k in
            ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    x = p["x"].to(DEV)
    ws = nv.ffn_workspace(1, 512)
    y = torch.empty(1, 1024, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nv.ffn_swiglu(*args, x, 1.0, workspace=ws, out=y)  # plan and tensor maps before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            nv.ffn_swiglu(*args, x, 1.0, workspace=ws, out=y)
    y.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    yr, ya, aux = reference(p, 1.0)
    assert_ffn_parity(y, yr, ya, aux, host(p["wd"]), host(p["sd"]), p["gd"], 1.0, "graph")
    assert not torch.any(ws[:HEADER])


def test_ffn_timeout_path_and_recovery():
    p = problem(1024, 512, 1, 880)
    nv.set_wait_budget_ns(0)
    run(p, 1.0)
    flags = nv.device_status()
    nv.set_wait_budget_ns(None)
    assert flags & nv.DEV_TIMEOUT
    check(p, 1.0, torch.float32, "after timeout")


def test_ffn_empty_and_invalid():
    p = problem(256, 256, 1, 890)
    args = [p[k].to(DEV) if torch.is_tensor(p[k]) else p[k] for k in
            ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    x = p["x"].to(DEV)
    y0 = nv.ffn_swiglu(*args, x[:0], 1.0)  # M = 0: nothing launched
    assert y0.shape == (0, 256)
    ws = nv.ffn_workspace(1, 256)
    with pytest.raises(nv.NVFP4Error):
        nv.ffn_swiglu(*args, x, 1.0, workspace=torch.zeros(ws.numel() + 16, dtype=torch.uint8, device=DEV)[16:])
    with pytest.raises(nv.NVFP4Error):
        nv.ffn_swiglu(*args, x, 0.0, workspace=ws)
    # I = 0: y = 0
    e = torch.empty(0, 128, dtype=torch.uint8, device=DEV)
    es = torch.empty(0, 16, dtype=torch.uint8, device=DEV)
    y = torch.full((1, 256), 7.0, device=DEV)
    nv.ffn_swiglu(e, es, 1.0, e, es, 1.0, torch.empty(256, 0, dtype=torch.uint8, device=DEV),
                  torch.empty(256, 0, dtype=torch.uint8, device=DEV), 1.0, x, 1.0, workspace=ws, out=y)
    torch.cuda.synchronize()
    assert not torch.any(y)
