"""GPU parity of the scale-dictionary GEMV (dense and routed experts) against the oracle.

The weights come from the generator's dictionary-constrained recipe (at most 32 scale codes per
tensor); the index plane and table are written by the generator's packer (synth.sdict_form,
pinned to a bit-by-bit packer in test_oracle_sdict; no library code), and the same bytes go to
the GPU and to the oracle. Tolerance as
in test_gpu_parity.py. Shapes: the attention projections and the 288-expert layer of
"glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json" (performance[64]: routed gate+up at 4.3125
bit/weight with a scale dictionary), the FFN down projection and ragged edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

from test_gpu_parity import DEV, assert_parity, host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_state():
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    yield
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    assert nv.device_status() == 0


def dense_case(N, K, M, seed, device="cpu"):
    p = synth.sdict_problem(N, K, M, seed, device=device)
    plane, table = synth.sdict_form(p["s"])
    return p, host(plane), host(table)


def run_dense(p, plane, table, out_dtype):
    y = nv.gemv_sdict(p["w"].to(DEV), torch.from_numpy(plane).to(DEV), torch.from_numpy(table).to(DEV), p["g"],
                      p["x"].to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    yr, ya = oracle.gemv_sdict(host(p["w"]), plane, table, p["g"], synth.bf16_bits(p["x"]))
    return y, yr, ya


@pytest.mark.parametrize("N,K,M,out", [(4096, 4096, 1, torch.bfloat16), (4096, 4096, 5, torch.bfloat16),
                                       (1024, 4096, 1, torch.bfloat16), (1024, 4096, 5, torch.float32),
                                       (4096, 12288, 1, torch.float32), (4096, 12288, 8, torch.float32)])
def test_workload_shapes(N, K, M, out):
    assert nv.describe_plan("dense_sdict", M, N, K).startswith("tile_sdict ")
    p, plane, table = dense_case(N, K, M, 700 + M, device=DEV)
    y, yr, ya = run_dense(p, plane, table, out)
    assert_parity(y, yr, ya, f"sdict {N}x{K} M={M}")


@pytest.mark.parametrize("M", range(1, 9))
@pytest.mark.parametrize("N,K", [(1000, 1024), (37, 2560), (300, 512), (1, 256), (513, 768)])
def test_m_sweep_ragged_rows(N, K, M):
    p, plane, table = dense_case(N, K, M, 710 + N + M)
    y, yr, ya = run_dense(p, plane, table, torch.float32 if M % 2 else torch.bfloat16)
    assert_parity(y, yr, ya, f"sdict {N}x{K} M={M}")


@pytest.mark.parametrize("variant", [1, 2, 3])
def test_other_kernels(variant):
    # 1: byte-load kernel, 2: tile kernel with exact fp32 x, 3: no tile kernel (byte-load runs)
    nv.set_variant(variant)
    for N, K, M in ((4096, 4096, 1), (300, 1024, 5)):
        p, plane, table = dense_case(N, K, M, 720 + variant)
        y, yr, ya = run_dense(p, plane, table, torch.float32)
        assert_parity(y, yr, ya, f"sdict variant {variant} {N}x{K} M={M}")


def test_random_indices_every_table_entry_and_extreme_codes():
    # indices drawn over the whole table, any non-NaN code (sign bit, subnormals, 448)
    N, K, M = 254, 1024, 3
    rng = np.random.default_rng(730)
    w = torch.from_numpy(rng.integers(0, 256, (N, K // 2), dtype=np.uint8))
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    table = rng.choice(codes, 32, replace=False).astype(np.uint8)
    table[0], table[1] = 0x01, 0x7E        # smallest subnormal, largest finite
    ind = rng.integers(0, 32, (N, K // 16))
    plane = synth.sdict_pack(torch.from_numpy(ind), N, K).numpy()
    x = synth.random_x(M, K, 731)
    p = {"w": w, "g": 0.5, "x": x}
    y, yr, ya = run_dense(p, plane, table, torch.float32)
    assert_parity(y, yr, ya, "sdict random indices")


def test_nan_table_entry_and_unaligned_plane():
    N, K, M = 200, 512, 2
    p, plane, table = dense_case(N, K, M, 740)
    table = table.copy()
    used = np.unique(host(p["s"]))
    table[len(used) - 1] = 0x7F             # the largest code used becomes NaN
    y, yr, ya = run_dense(p, plane, table, torch.float32)
    assert np.isnan(yr).any() and not np.isnan(yr).all()
    assert_parity(y, yr, ya, "sdict nan entry")
    # an index plane that is not 16-byte aligned runs the byte-load kernel
    buf = torch.zeros(plane.size + 1, dtype=torch.uint8, device=DEV)
    buf[1:] = torch.from_numpy(plane).to(DEV)
    y2 = nv.gemv_sdict(p["w"].to(DEV), buf[1:], torch.from_numpy(table).to(DEV), p["g"], p["x"].to(DEV))
    torch.cuda.synchronize()
    assert_parity(y2, yr, ya, "sdict unaligned plane")


def moe_case(T, x_per_slot, seed):
    N, K = (4096, 1536) if x_per_slot else (3072, 4096)
    p = synth.moe_problem(288, N, K, T, 8, x_per_slot, seed=seed, device=DEV, max_codes=32)
    s = host(p["s"])
    routed = sorted(set(host(p["ids"]).tolist()))
    planes = np.zeros((288, nv.sdict_plane_bytes(N, K)), dtype=np.uint8)
    tables = np.zeros((288, 32), dtype=np.uint8)
    for e in routed:
        pl, tb = synth.sdict_form(torch.from_numpy(s[e]))
        planes[e], tables[e] = pl.numpy(), tb.numpy()
    return p, planes, tables


@pytest.mark.parametrize("T", [4, 16])
@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_288_experts_top8(x_per_slot, T):
    p, planes, tables = moe_case(T, x_per_slot, 750 + T)
    N, K = p["N"], p["K"]
    kind = "moe_per_slot_sdict" if x_per_slot else "moe_sdict"
    want = "tile_sk_moe_sdict"  # up to 256 slots, group-aligned stream-K
    assert nv.describe_plan(kind, 288, N, K, T, 8).split()[0] == want
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv_sdict(p["w"], torch.from_numpy(planes).to(DEV), torch.from_numpy(tables).to(DEV), p["gs"],
                          p["ids"], p["x"], x_per_slot, 8, out_dtype=torch.bfloat16 if T == 4 else torch.float32,
                          status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yr, ya, bad = oracle.moe_gemv_sdict(host(p["w"]), planes, tables, host(p["gs"]), host(p["ids"]),
                                        synth.bf16_bits(p["x"]), x_per_slot, 8)
    assert bad == 0
    assert_parity(y, yr, ya, f"moe sdict T={T} {want}")


def test_moe_timeout_path_and_recovery():
    p, planes, tables = moe_case(4, False, 760)
    args = (p["w"], torch.from_numpy(planes).to(DEV), torch.from_numpy(tables).to(DEV), p["gs"], p["ids"], p["x"],
            False, 8)
    nv.set_wait_budget_ns(0)
    nv.moe_gemv_sdict(*args)
    flags = nv.device_status()
    nv.set_wait_budget_ns(None)
    assert flags & nv.DEV_TIMEOUT
    y = nv.moe_gemv_sdict(*args)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    yr, ya, _ = oracle.moe_gemv_sdict(host(p["w"]), planes, tables, host(p["gs"]), host(p["ids"]),
                                      synth.bf16_bits(p["x"]), False, 8)
    assert_parity(y, yr, ya, "moe sdict after timeout")
