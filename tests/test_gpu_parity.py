"""GPU parity: the CUDA kernels (called through the C ABI) against the CPU oracle.

Tolerance, per output element, with A = |g| * sum_k |w_k x_k| from the oracle:
  fp32 output:  |y - y_ref| <= 1e-5 * A + 1e-6
  bf16 output:  the same bound plus one bf16 ulp of y_ref
y_ref is the oracle's fp64 value (not rounded). NaN must appear exactly where the oracle
has NaN. Inputs are seeded (generator module). Large cases generate on the GPU with torch's
CUDA RNG and copy the bytes to the host for the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def assert_parity(y_gpu: torch.Tensor, y_ref: np.ndarray, yabs: np.ndarray, what: str = ""):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan_ref), f"{what}: NaN positions differ"
    tol = 1e-5 * yabs + 1e-6
    if y_gpu.dtype == torch.bfloat16:
        tol = tol + ulp_bf16(y_ref)
    err = np.where(nan_ref, 0.0, np.abs(y - y_ref))
    bad = err > np.where(nan_ref, 1.0, tol)
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={y[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")


def host(t):
    return t.detach().cpu().numpy()


def run_dense(N, K, M, seed, out_dtype, device="cpu"):
    p = synth.dense_problem(N, K, M, seed, device=device)
    w, s, x = (p[k].to(DEV) for k in ("w", "s", "x"))
    y = nv.gemv(w, s, p["g"], x, out_dtype=out_dtype)
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    return y, yr, ya


@pytest.fixture(autouse=True)
def _clean_state():
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    yield
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    assert nv.device_status() == 0


# ------------------------------------------------------------------ workload configs

def test_smoke_256x512_m1_fp32():
    y, yr, ya = run_dense(256, 512, 1, 0, torch.float32)
    assert_parity(y, yr, ya, "256x512 M=1")


@pytest.mark.parametrize("N,K,M,seed", [(4096, 4096, 1, 1), (4096, 4096, 5, 2),
                                        (1024, 4096, 1, 3), (1024, 4096, 5, 4)])
def test_attention_projections_bf16(N, K, M, seed):
    y, yr, ya = run_dense(N, K, M, seed, torch.bfloat16)
    assert_parity(y, yr, ya, f"{N}x{K} M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_ffn_gate_up_fused(M):
    N, K = 12288, 4096
    p = synth.gate_up_problem(N, K, M, 5, device=DEV)
    y = nv.gemv_gate_up(p["wg"], p["sg"], p["gg"], p["wu"], p["su"], p["gu"], p["x"])
    torch.cuda.synchronize()
    yr, ya = oracle.gemv_gate_up(host(p["wg"]), host(p["sg"]), p["gg"], host(p["wu"]), host(p["su"]),
                                 p["gu"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, f"gate_up M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_ffn_down(M):
    y, yr, ya = run_dense(4096, 12288, M, 6, torch.float32, device=DEV)
    assert_parity(y, yr, ya, f"down M={M}")


def test_vocab_head_m1():
    y, yr, ya = run_dense(151936, 4096, 1, 7, torch.float32, device=DEV)
    assert_parity(y, yr, ya, "vocab head")


@pytest.mark.parametrize("variant", [0, 3])
@pytest.mark.parametrize("x_per_slot,N,K", [(False, 3072, 4096), (True, 4096, 1536)])
def test_moe_288_experts_top8(x_per_slot, N, K, variant):
    # variant 3: the bulk-copy streaming kernel instead of the warp-tile kernel
    nv.set_variant(variant)
    p = synth.moe_problem(288, N, K, 4, 8, x_per_slot, seed=8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], x_per_slot, 8, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]),
                                  synth.bf16_bits(p["x"]), x_per_slot, 8)
    assert bad == 0
    assert_parity(y, yr, ya, "moe")


# ------------------------------------------------------------------ shapes, tails, edge cases

@pytest.mark.parametrize("M", range(1, 9))
@pytest.mark.parametrize("N,K", [(1000, 1056), (37, 2816), (300, 512)])
def test_m_sweep_ragged(N, K, M):
    y, yr, ya = run_dense(N, K, M, 100 + M, torch.float32)
    assert_parity(y, yr, ya, f"{N}x{K} M={M}")


@pytest.mark.parametrize("N,K,M", [(1, 16, 1), (3, 48, 2), (33, 80, 3), (5, 32, 8), (1, 32, 1),
                                   (7, 1040, 1), (2, 16, 8), (513, 32, 4)])
def test_small_and_odd_shapes(N, K, M):
    for dt in (torch.float32, torch.bfloat16):
        y, yr, ya = run_dense(N, K, M, 200 + N + K + M, dt)
        assert_parity(y, yr, ya, f"{N}x{K} M={M} {dt}")


@pytest.mark.parametrize("N,K,M", [(1000, 1024, 1), (1000, 1024, 3), (37, 2560, 8), (513, 768, 2),
                                   (1, 256, 1), (5, 256, 7), (4096, 768, 4), (300, 12288, 1), (2000, 2048, 6)])
def test_tile_kernel_ragged_rows(N, K, M):
    # K % 256 == 0 runs the warp-tile kernel; N % 16 != 0 leaves zero-filled rows in the last tile
    assert nv.describe_plan("dense", M, N, K).startswith("tile ")
    for dt in (torch.float32, torch.bfloat16):
        y, yr, ya = run_dense(N, K, M, 400 + N + K + M, dt)
        assert_parity(y, yr, ya, f"{N}x{K} M={M} {dt}")


@pytest.mark.parametrize("N,K,M", [(4096, 4096, 1), (1024, 4096, 5), (4096, 12288, 2), (256, 512, 1)])
def test_stream_kernel_on_tile_shapes(N, K, M):
    # the bulk-copy streaming kernel stays correct on shapes the tile kernel normally takes
    nv.set_variant(3)
    assert nv.describe_plan("dense", M, N, K).startswith("stream ")
    y, yr, ya = run_dense(N, K, M, 500 + M, torch.bfloat16, device=DEV)
    assert_parity(y, yr, ya, f"stream {N}x{K} M={M}")
    p = synth.gate_up_problem(2000, 2048, 3, 307, device=DEV)
    y = nv.gemv_gate_up(p["wg"], p["sg"], p["gg"], p["wu"], p["su"], p["gu"], p["x"])
    torch.cuda.synchronize()
    yr, ya = oracle.gemv_gate_up(host(p["wg"]), host(p["sg"]), p["gg"], host(p["wu"]), host(p["su"]),
                                 p["gu"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "stream gate_up")


def test_empty_inputs():
    w = torch.empty(0, 8, dtype=torch.uint8, device=DEV)
    s = torch.empty(0, 1, dtype=torch.uint8, device=DEV)
    x = torch.zeros(2, 16, dtype=torch.bfloat16, device=DEV)
    assert nv.gemv(w, s, 1.0, x).shape == (2, 0)
    p = synth.dense_problem(8, 32, 1, 300)
    w, s = p["w"].to(DEV), p["s"].to(DEV)
    x0 = torch.zeros(0, 32, dtype=torch.bfloat16, device=DEV)
    assert nv.gemv(w, s, p["g"], x0).shape == (0, 8)
    # K == 0: empty sum
    wk = torch.empty(4, 0, dtype=torch.uint8, device=DEV)
    sk = torch.empty(4, 0, dtype=torch.uint8, device=DEV)
    xk = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    y = nv.gemv(wk, sk, 1.0, xk, out=torch.full((3, 4), 7.0, device=DEV))
    assert torch.all(y == 0)


def test_unaligned_pointers_use_byte_kernel():
    N, K, M = 64, 256, 2
    p = synth.dense_problem(N, K, M, 301)
    wbuf = torch.zeros(N * K // 2 + 1, dtype=torch.uint8, device=DEV)
    sbuf = torch.zeros(N * K // 16 + 1, dtype=torch.uint8, device=DEV)
    wbuf[1:] = p["w"].reshape(-1).to(DEV)
    sbuf[1:] = p["s"].reshape(-1).to(DEV)
    w = wbuf[1:].view(N, K // 2)
    s = sbuf[1:].view(N, K // 16)
    assert w.data_ptr() % 16 == 1
    y = nv.gemv(w, s, p["g"], p["x"].to(DEV))
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "unaligned")


def test_unaligned_scale_rows_tma_head_tail():
    # K % 256 != 0: scale rows are not 16-byte multiples, so items start mid-line
    for N, K, M in ((777, 704, 2), (129, 1120, 1), (50, 96, 3)):
        y, yr, ya = run_dense(N, K, M, 302 + K, torch.float32)
        assert_parity(y, yr, ya, f"{N}x{K}")


def test_nan_scale_propagates():
    N, K, M = 300, 512, 2
    p = synth.dense_problem(N, K, M, 303)
    s = p["s"].clone()
    s[17, 3] = 0x7F
    s[299, 31] = 0xFF
    y = nv.gemv(p["w"].to(DEV), s.to(DEV), p["g"], p["x"].to(DEV))
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(s), p["g"], synth.bf16_bits(p["x"]))
    assert np.isnan(yr[:, 17]).all() and np.isnan(yr[:, 299]).all()
    assert_parity(y, yr, ya, "nan scales")


def test_sign_bit_scales_and_extreme_codes():
    # every E4M3 scale code except NaN, every E2M1 code, large and tiny x
    N, K, M = 254, 512, 2
    g = torch.Generator().manual_seed(304)
    w = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=g)
    codes = torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8)
    s = codes[torch.randint(0, codes.numel(), (N, K // 16), generator=g)]
    x = (torch.randn(M, K, generator=g) * torch.exp2(torch.randint(-20, 20, (M, K), generator=g).float())
         ).to(torch.bfloat16)
    y = nv.gemv(w.to(DEV), s.to(DEV), 0.75, x.to(DEV))
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(w.numpy(), s.numpy(), 0.75, synth.bf16_bits(x))
    assert_parity(y, yr, ya, "extreme codes")


def test_non_finite_x_matches_oracle():
    # Inf in x: the f16 staging reports it and the CTA falls back to the fp32 path
    N, K, M = 200, 1024, 2
    p = synth.dense_problem(N, K, M, 308)
    x = p["x"].clone()
    x[0, 5] = float("inf")
    x[1, 700] = float("-inf")
    y = nv.gemv(p["w"].to(DEV), p["s"].to(DEV), p["g"], x.to(DEV))
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(x))
    yg = y.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(yg), np.isnan(yr))
    assert np.array_equal(np.isinf(yg), np.isinf(yr)) and np.array_equal(yg[np.isinf(yr)], yr[np.isinf(yr)])
    fin = np.isfinite(yr)
    assert np.all(np.abs(yg[fin] - yr[fin]) <= 1e-5 * ya[fin] + 1e-6)


def test_normal_x_stays_on_f16_path_and_fp32_variant_matches():
    nv.fp32_fallbacks()
    y, yr, ya = run_dense(2048, 4096, 2, 340, torch.float32, device=DEV)
    assert_parity(y, yr, ya, "f16 path")
    assert nv.fp32_fallbacks() == 0
    nv.set_variant(2)
    y, yr, ya = run_dense(2048, 4096, 2, 340, torch.float32, device=DEV)
    assert_parity(y, yr, ya, "fp32 path")


def test_wide_dynamic_range_x_uses_exact_path():
    # x spans 2^-60..2^60 inside 16-element blocks, so block-scaled f16 cannot hold it
    N, K = 300, 2048
    nv.fp32_fallbacks()
    for M in (1, 2, 4):
        p = synth.dense_problem(N, K, M, 309 + M)
        g = torch.Generator().manual_seed(M)
        x = (p["x"].float() * torch.exp2(torch.randint(-60, 60, (M, K), generator=g).float())).to(torch.bfloat16)
        y = nv.gemv(p["w"].to(DEV), p["s"].to(DEV), p["g"], x.to(DEV))
        torch.cuda.synchronize()
        yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(x))
        assert_parity(y, yr, ya, f"wide range M={M}")
        assert nv.fp32_fallbacks() > 0


@pytest.mark.parametrize("pdl", [True, False])
def test_chained_gemvs_back_to_back(pdl):
    # each call's bf16 output is the next call's x, launched back to back on one stream: the
    # dependent kernel must read x only after its producer finished
    nv.set_pdl(pdl)
    try:
        M, dims = 3, [4096, 2048, 4096, 1024, 4096, 512]
        probs = [synth.dense_problem(dims[i + 1], dims[i], M, 330 + i, device=DEV) for i in range(len(dims) - 1)]
        x0 = synth.random_x(M, dims[0], 339, device=DEV)
        xs = [x0]
        for _ in range(3):
            xs = [x0]
            for q in probs:
                xs.append(nv.gemv(q["w"], q["s"], q["g"], xs[-1], out_dtype=torch.bfloat16))
        torch.cuda.synchronize()
        for i, q in enumerate(probs):
            yr, ya = oracle.gemv(host(q["w"]), host(q["s"]), q["g"], synth.bf16_bits(xs[i]))
            assert_parity(xs[i + 1], yr, ya, f"chain step {i}")
    finally:
        nv.set_pdl(True)


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_fp32_variant_on_configs(M):
    nv.set_variant(2)
    y, yr, ya = run_dense(4096, 4096, M, 341 + M, torch.bfloat16, device=DEV)
    assert_parity(y, yr, ya, f"fp32 x M={M}")
    p = synth.moe_problem(64, 512, 1024, 3, 4, True, seed=345, fill="all")
    st, _ = _moe_check(p, p["ids"].tolist(), True, 4)
    assert st == 0


def test_byte_kernel_matches_oracle_on_configs():
    nv.set_variant(1)
    for N, K, M, dt in ((4096, 4096, 1, torch.bfloat16), (1024, 4096, 5, torch.bfloat16),
                        (300, 12288, 8, torch.float32)):
        y, yr, ya = run_dense(N, K, M, 305, dt)
        assert_parity(y, yr, ya, f"byte kernel {N}x{K} M={M}")


def test_deterministic_across_runs():
    p = synth.dense_problem(4096, 12288, 4, 306, device=DEV)
    ys = [nv.gemv(p["w"], p["s"], p["g"], p["x"]) for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


def test_gate_up_matches_two_dense_calls():
    # the fused launch may split rows and K differently (another fp32 summation order), so
    # both are held to the oracle's tolerance rather than to bitwise equality
    p = synth.gate_up_problem(2000, 2048, 3, 307, device=DEV)
    y = nv.gemv_gate_up(p["wg"], p["sg"], p["gg"], p["wu"], p["su"], p["gu"], p["x"])
    yg = nv.gemv(p["wg"], p["sg"], p["gg"], p["x"])
    yu = nv.gemv(p["wu"], p["su"], p["gu"], p["x"])
    torch.cuda.synchronize()
    yr, ya = oracle.gemv_gate_up(host(p["wg"]), host(p["sg"]), p["gg"], host(p["wu"]), host(p["su"]),
                                 p["gu"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "fused")
    assert_parity(torch.cat([yg, yu], 1), yr, ya, "two dense calls")


# ------------------------------------------------------------------ MoE edge cases

def _moe_check(p, ids, x_per_slot, top_k, out_dtype=torch.float32):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idd = torch.as_tensor(ids, dtype=torch.int32).to(DEV)
    y = nv.moe_gemv(p["w"].to(DEV), p["s"].to(DEV), p["gs"].to(DEV), idd, p["x"].to(DEV), x_per_slot,
                    top_k, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), np.asarray(ids, np.int32),
                                  synth.bf16_bits(p["x"]), x_per_slot, top_k)
    assert_parity(y, yr, ya, "moe")
    return int(st.item()), bad


@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_repeated_experts_are_shared(x_per_slot):
    E, N, K, T, top_k = 16, 200, 1024, 5, 3
    p = synth.moe_problem(E, N, K, T, top_k, x_per_slot, seed=310, fill="all")
    ids = [3, 3, 7, 3, 9, 7, 3, 3, 3, 1, 3, 5, 0, 3, 15]   # expert 3 in 8 slots (> one group)
    st, bad = _moe_check(p, ids, x_per_slot, top_k)
    assert st == 0 and bad == 0


@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_tile_groups_32_slots(x_per_slot):
    # 32 slots (the tile kernel's limit): one expert in 20 slots (three groups of <= 8), the
    # rest spread, a ragged N and bf16 output
    E, N, K, T, top_k = 12, 200, 1024, 4, 8
    p = synth.moe_problem(E, N, K, T, top_k, x_per_slot, seed=315, fill="all")
    ids = [5] * 20 + [0, 1, 2, 3, 4, 6, 7, 8, 9, 10, 11, 1]
    assert nv.describe_plan("moe_per_slot" if x_per_slot else "moe", E, N, K, T, top_k).split()[0] in (
        "tile_moe", "tile_sk_moe")
    st, bad = _moe_check(p, ids, x_per_slot, top_k, torch.bfloat16)
    assert st == 0 and bad == 0


@pytest.mark.parametrize("x_per_slot,N,K,E,T,top_k", [(False, 3072, 4096, 288, 4, 8), (True, 4096, 1536, 288, 4, 8),
                                                       (True, 200, 1024, 7, 5, 3), (False, 512, 1024, 40, 2, 6)])
def test_moe_stream_k(x_per_slot, N, K, E, T, top_k):
    # the stream-K MoE form: jobs (expert group, tile) spread evenly over the CTAs and TMA boxes
    # over the warps, with tiles that straddle warps combined through shared memory
    assert nv.describe_plan("moe_per_slot" if x_per_slot else "moe", E, N, K, T, top_k).split()[0] == "tile_sk_moe"
    # only the routed experts are filled (the rest stay zero): generated on the device
    p = synth.moe_problem(E, N, K, T, top_k, x_per_slot, seed=316 + N, device=DEV)
    st, bad = _moe_check(p, p["ids"].tolist(), x_per_slot, top_k, torch.bfloat16)
    assert st == 0 and bad == 0


def test_moe_bad_ids_zero_their_rows():
    E, N, K, T, top_k = 6, 96, 512, 2, 3
    p = synth.moe_problem(E, N, K, T, top_k, True, seed=311, fill="all")
    ids = [0, -2, 5, 6, 1, 1]
    st, bad = _moe_check(p, ids, True, top_k, torch.bfloat16)
    assert bad == 2 and st & nv.DEV_BAD_EXPERT
    assert nv.device_status() & nv.DEV_BAD_EXPERT


def test_moe_byte_kernel_and_many_slots():
    E, N, K = 40, 64, 256
    p = synth.moe_problem(E, N, K, 100, 3, False, seed=312, fill="all")   # 300 slots > 256
    st, bad = _moe_check(p, p["ids"].tolist(), False, 3)
    assert st == 0
    nv.set_variant(1)
    q = synth.moe_problem(E, N, K, 4, 8, True, seed=313, fill="all")
    st, bad = _moe_check(q, q["ids"].tolist(), True, 8)
    assert st == 0


def test_moe_odd_k_uses_byte_kernel():
    p = synth.moe_problem(10, 33, 48, 3, 2, False, seed=314, fill="all")
    st, _ = _moe_check(p, p["ids"].tolist(), False, 2)
    assert st == 0


# ------------------------------------------------------------------ runtime behaviour

@pytest.mark.parametrize("variant", [0, 3])
def test_timeout_path_reports_and_recovers(variant):
    # a zero wait budget makes the pipeline waits give up: the kernel must report it, drain its
    # copies and leave the context usable (variant 3: the bulk-copy streaming kernel)
    nv.set_variant(variant)
    p = synth.dense_problem(4096, 4096, 1, 320, device=DEV)
    nv.set_wait_budget_ns(0)
    nv.gemv(p["w"], p["s"], p["g"], p["x"])
    flags = nv.device_status()
    nv.set_wait_budget_ns(None)
    assert flags & nv.DEV_TIMEOUT
    y = nv.gemv(p["w"], p["s"], p["g"], p["x"])
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "after timeout")


def test_cuda_graph_capture_and_replay():
    p = synth.dense_problem(2048, 4096, 2, 321, device=DEV)
    y = torch.empty(2, 2048, device=DEV)
    nv.gemv(p["w"], p["s"], p["g"], p["x"], out=y)     # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            nv.gemv(p["w"], p["s"], p["g"], p["x"], out=y)
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "graph replay")


def test_side_stream_launch():
    p = synth.dense_problem(1024, 2048, 3, 322, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = nv.gemv(p["w"], p["s"], p["g"], p["x"])
    s.synchronize()
    yr, ya = oracle.gemv(host(p["w"]), host(p["s"]), p["g"], synth.bf16_bits(p["x"]))
    assert_parity(y, yr, ya, "side stream")


def test_plan_uses_all_sms_for_large_problems():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    desc = nv.describe_plan("dense", 1, 151936, 4096)
    grid = int(desc.split("grid=")[1].split()[0])
    assert desc.split()[0] in ("tile", "stream") and grid % sms == 0 and grid >= sms
    desc = nv.describe_plan("dense", 8, 4096, 12288)
    assert "split=" in desc and "split=1 " not in desc


# ------------------------------------------------------------------ fused gate/up activation
# y = silu(c(gate)) * c(up), c = clamp to [-lim, lim]. The GPU's gate and up carry the GEMV
# tolerance tg = 1e-5 * A_gate + 1e-6 (tu likewise); the clamp does not enlarge an error,
# |silu'| <= 1.1 everywhere and |silu(v)| <= max(|v|, 0.28), so an output may differ by
#   1.1 * |c(up)| * tg + max(|c(gate)|, 0.28) * tu + 1.1 * tg * tu
# plus the fp32 evaluation of the activation (a few roundings and expf: 1e-6 * |y|), the
# absolute 1e-6, and one bf16 ulp of y_ref for bf16 output.

def swiglu_tolerance(aux, y_ref, lim, bf16):
    tg = 1e-5 * aux["gate_abs"] + 1e-6
    tu = 1e-5 * aux["up_abs"] + 1e-6
    cg = np.clip(aux["gate"], -lim, lim)
    cu = np.clip(aux["up"], -lim, lim)
    tol = 1.1 * np.abs(cu) * tg + np.maximum(np.abs(cg), 0.28) * tu + 1.1 * tg * tu
    tol = tol + 1e-6 * np.abs(np.nan_to_num(y_ref)) + 1e-6
    if bf16:
        tol = tol + ulp_bf16(np.nan_to_num(y_ref))
    return tol


def assert_swiglu_parity(y_gpu, y_ref, aux, lim, what=""):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan_ref), f"{what}: NaN positions differ"
    tol = swiglu_tolerance(aux, y_ref, lim, y_gpu.dtype == torch.bfloat16)
    err = np.where(nan_ref, 0.0, np.abs(y - y_ref))
    bad = err > np.where(nan_ref, 1.0, tol)
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={y[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")


def run_swiglu(N, K, M, seed, lim, out_dtype, device="cpu", p=None):
    p = p or synth.gate_up_problem(N, K, M, seed, device=device)
    wg, sg, wu, su, x = (p[k].to(DEV) for k in ("wg", "sg", "wu", "su", "x"))
    y = nv.gemv_gate_up_swiglu(wg, sg, p["gg"], wu, su, p["gu"], x, lim, out_dtype=out_dtype)
    torch.cuda.synchronize()
    yr, aux = oracle.gate_up_swiglu(host(p["wg"]), host(p["sg"]), p["gg"], host(p["wu"]), host(p["su"]),
                                    p["gu"], synth.bf16_bits(p["x"]), lim)
    return y, yr, aux


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("lim", [math.inf, 1.0])
def test_swiglu_ffn_shape(M, lim):
    # the FFN gate/up projection (2 x 12288 x 4096); lim = 1 clamps part of gate and up
    y, yr, aux = run_swiglu(12288, 4096, M, 5, lim, torch.bfloat16, device=DEV)
    if lim < math.inf:
        assert (np.abs(aux["gate"]) > lim).any() and (np.abs(aux["up"]) > lim).any()
    assert_swiglu_parity(y, yr, aux, lim, f"swiglu ffn M={M} lim={lim}")


@pytest.mark.parametrize("N,K,M", [(3072, 4096, 4), (4096, 4096, 8), (1000, 1024, 3), (37, 2560, 8),
                                   (513, 768, 2), (1, 256, 1), (5, 256, 7), (300, 12288, 1),
                                   (2000, 2048, 8), (4096, 1536, 5)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_swiglu_tile_plans_and_ragged_rows(N, K, M, out):
    # plans with a K split over warps, over a cluster (S = 4 and 8), one warp per tile, and
    # N not a multiple of 16
    y, yr, aux = run_swiglu(N, K, M, 600 + N % 97 + M, 0.5, out)
    assert_swiglu_parity(y, yr, aux, 0.5, f"swiglu {N}x{K} M={M}")


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_swiglu_other_kernels(variant):
    # 1: byte-load kernel; 2: tile kernel in exact fp32; 3: streaming kernel requested (the
    # fused form has no streaming instantiation, so the byte-load kernel runs)
    nv.set_variant(variant)
    for N, K, M in ((300, 512, 1), (129, 1024, 5)):
        y, yr, aux = run_swiglu(N, K, M, 640 + variant, 0.75, torch.float32)
        assert_swiglu_parity(y, yr, aux, 0.75, f"swiglu variant {variant} {N}x{K}")


@pytest.mark.parametrize("N,K,M", [(77, 528, 3), (40, 96, 1), (3, 16, 8)])
def test_swiglu_k_not_multiple_of_256(N, K, M):
    y, yr, aux = run_swiglu(N, K, M, 650 + K, 2.0, torch.bfloat16)
    assert_swiglu_parity(y, yr, aux, 2.0, f"swiglu {N}x{K}")


def test_swiglu_and_gate_up_agree_with_the_oracle_on_the_same_inputs():
    # the fused call and the unfused gate_up call on the same weights and x, each against the
    # oracle: gate_up against the oracle's gate and up (GEMV tolerance), the fused output against
    # the oracle's activation of them (SwiGLU tolerance)
    p = synth.gate_up_problem(2048, 4096, 2, 660, device=DEV)
    yf = nv.gemv_gate_up_swiglu(p["wg"], p["sg"], p["gg"], p["wu"], p["su"], p["gu"], p["x"], 1.5,
                                out_dtype=torch.float32)
    gu = nv.gemv_gate_up(p["wg"], p["sg"], p["gg"], p["wu"], p["su"], p["gu"], p["x"])
    torch.cuda.synchronize()
    args = (host(p["wg"]), host(p["sg"]), p["gg"], host(p["wu"]), host(p["su"]), p["gu"], synth.bf16_bits(p["x"]))
    yr, aux = oracle.gate_up_swiglu(*args, 1.5)
    assert_parity(gu, np.concatenate([aux["gate"], aux["up"]], 1),
                  np.concatenate([aux["gate_abs"], aux["up_abs"]], 1), "gate_up beside the fused call")
    assert_swiglu_parity(yf, yr, aux, 1.5, "fused SwiGLU beside gate_up")


def test_swiglu_nan_scale_and_empty_inputs():
    N, K, M = 300, 512, 2
    p = synth.gate_up_problem(N, K, M, 670)
    sg = p["sg"].clone()
    sg[17, 3] = 0x7F                      # NaN gate in row 17
    su = p["su"].clone()
    su[200, 0] = 0xFF                     # NaN up in row 200
    q = dict(p, sg=sg, su=su)
    y, yr, aux = run_swiglu(N, K, M, 0, 1.0, torch.float32, p=q)
    assert np.isnan(yr[:, 17]).all() and np.isnan(yr[:, 200]).all()
    assert_swiglu_parity(y, yr, aux, 1.0, "swiglu nan")
    # K = 0: gate = up = 0, so y = 0; M = 0 and N = 0 launch nothing
    z = torch.empty(4, 0, dtype=torch.uint8, device=DEV)
    x0 = torch.empty(2, 0, dtype=torch.bfloat16, device=DEV)
    y0 = torch.full((2, 4), 7.0, device=DEV)
    nv.gemv_gate_up_swiglu(z, z, 1.0, z, z, 1.0, x0, out=y0)
    torch.cuda.synchronize()
    assert torch.all(y0 == 0)
    assert nv.describe_plan("gate_up_swiglu", 1, 12288, 4096).startswith("tile_swiglu ")
    assert nv.describe_plan("gate_up_swiglu", 1, 100, 528).startswith("simple ")


def test_graph_of_a_step_with_host_copies():
    # one captured step: pinned x -> device, a fused gate/up + SwiGLU call and a MoE call
    # (PDL-chained), y -> pinned host; replayed with new host inputs each time
    q = synth.gate_up_problem(512, 1024, 2, 323, device=DEV)
    r = synth.moe_problem(16, 256, 512, 2, 4, True, seed=324, device=DEV, fill="all")
    hx1 = torch.empty(2, 1024, dtype=torch.bfloat16).pin_memory()
    hx2 = torch.empty(8, 512, dtype=torch.bfloat16).pin_memory()
    hy1 = torch.empty(2, 512, dtype=torch.bfloat16).pin_memory()
    hy2 = torch.empty(8, 256).pin_memory()
    dx1, dx2 = torch.empty(2, 1024, dtype=torch.bfloat16, device=DEV), torch.empty(8, 512, dtype=torch.bfloat16, device=DEV)
    y1, y2 = torch.empty(2, 512, dtype=torch.bfloat16, device=DEV), torch.empty(8, 256, device=DEV)

    def step():
        dx1.copy_(hx1, non_blocking=True)
        dx2.copy_(hx2, non_blocking=True)
        nv.gemv_gate_up_swiglu(q["wg"], q["sg"], q["gg"], q["wu"], q["su"], q["gu"], dx1, 0.5, out=y1)
        nv.moe_gemv(r["w"], r["s"], r["gs"], r["ids"], dx2, True, 4, out=y2)
        hy1.copy_(y1, non_blocking=True)
        hy2.copy_(y2, non_blocking=True)

    step()  # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (325, 326):
        x1 = synth.random_x(2, 1024, seed)
        x2 = synth.random_x(8, 512, seed + 100)
        hx1.copy_(x1)
        hx2.copy_(x2)
        graph.replay()
        torch.cuda.synchronize()
        yr, aux = oracle.gate_up_swiglu(host(q["wg"]), host(q["sg"]), q["gg"], host(q["wu"]), host(q["su"]),
                                        q["gu"], synth.bf16_bits(x1), 0.5)
        assert_swiglu_parity(hy1, yr, aux, 0.5, "graph swiglu")
        ym, ya, _ = oracle.moe_gemv(host(r["w"]), host(r["s"]), host(r["gs"]), host(r["ids"]),
                                    synth.bf16_bits(x2), True, 4)
        assert_parity(hy2, ym, ya, "graph moe")
