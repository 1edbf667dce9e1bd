"""GPU parity of the routed-expert GEMV at larger routings (33..256 slots), with hot experts
routed to more than 8 and more than 16 slots, and the timeout path of the tile kernels' MoE
forms. Same tolerance as test_gpu_parity.py (shared helpers imported from there).

Shapes are the 288-expert layer of "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json"
(performance[33], routed gate or up; performance[64], the routed gate+up union): gate_up
[3072, 4096] with x shared by a token's slots, down [4096, 1536] with one x row per slot.
"""
import numpy as np
import pytest
import torch

import oracle
import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

from test_gpu_parity import DEV, assert_parity, host

pytestmark = pytest.mark.gpu

E, TOP_K = 288, 8
SHAPES = {False: (3072, 4096), True: (4096, 1536)}  # x_per_slot -> (N, K)


@pytest.fixture(autouse=True)
def _clean_state():
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    yield
    nv.set_variant(0)
    nv.set_wait_budget_ns(None)
    assert nv.device_status() == 0


_cache = {}


def problem(T, x_per_slot, ids=None, tag="seeded"):
    """One generated problem and its oracle result, shared by the kernel variants."""
    key = (T, x_per_slot, tag)
    if key not in _cache:
        _cache.clear()  # one problem on the device at a time (the expert tensors are GBs)
        N, K = SHAPES[x_per_slot]
        p = synth.moe_problem(E, N, K, T, TOP_K, x_per_slot, seed=900 + T, device=DEV, ids=ids)
        yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]),
                                      synth.bf16_bits(p["x"]), x_per_slot, TOP_K)
        assert bad == 0
        _cache[key] = (p, yr, ya)
    return _cache[key]


def run(p, x_per_slot, out_dtype):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], x_per_slot, TOP_K, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y


def plan_kernel(T, x_per_slot):
    N, K = SHAPES[x_per_slot]
    return nv.describe_plan("moe_per_slot" if x_per_slot else "moe", E, N, K, T, TOP_K).split()[0]


@pytest.mark.parametrize("variant", [0, 3])
@pytest.mark.parametrize("x_per_slot", [False, True])
@pytest.mark.parametrize("T", [5, 16, 32])
def test_moe_many_slots(T, x_per_slot, variant):
    # 40..256 slots: beyond the 32 slots of the tile kernels' first form. variant 3 forces the
    # bulk-copy streaming kernel; variant 0 takes the library's own choice.
    nv.set_variant(variant)
    kern = plan_kernel(T, x_per_slot)
    if variant == 3:
        assert kern == "stream_moe", kern
    else:
        assert kern in ("stream_moe", "tile_moe", "tile_sk_moe"), kern
    p, yr, ya = problem(T, x_per_slot)
    out = torch.bfloat16 if T == 16 else torch.float32
    y = run(p, x_per_slot, out)
    assert_parity(y, yr, ya, f"moe T={T} x_per_slot={x_per_slot} {kern}")


def hot_routing(T, seed):
    """T tokens x top-8 distinct experts, with expert 5 in the first 12 tokens, 9 in the first
    20 and 11 in every token (T = 32: 12, 20 and 32 slots, i.e. 2, 3 and 4 groups of at most
    8), the other ids seeded."""
    forced = [(5, 12), (9, 20), (11, T)]
    fset = {e for e, _ in forced}
    ids = synth.routing(T, TOP_K, E, seed).view(T, TOP_K).clone()
    for t in range(T):
        want = [e for e, n in forced if t < n]
        rest = [v for v in ids[t].tolist() if v not in fset]
        c = 0
        while len(rest) < TOP_K - len(want):  # refill with experts the token does not use yet
            if c not in fset and c not in rest:
                rest.append(c)
            c += 1
        ids[t] = torch.tensor(want + rest[:TOP_K - len(want)], dtype=torch.int32)
    ids = ids.reshape(-1)
    for t in range(T):
        assert len(set(ids[t * TOP_K:(t + 1) * TOP_K].tolist())) == TOP_K
    return ids


@pytest.mark.parametrize("variant", [0, 3])
@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_hot_experts_beyond_8_and_16_slots(x_per_slot, variant):
    nv.set_variant(variant)
    T = 32
    ids = hot_routing(T, 931)
    counts = np.bincount(ids.numpy(), minlength=E)
    assert counts[5] == 12 and counts[9] == 20 and counts[11] == 32
    p, yr, ya = problem(T, x_per_slot, ids=ids, tag="hot")
    y = run(p, x_per_slot, torch.float32)
    assert_parity(y, yr, ya, f"hot experts x_per_slot={x_per_slot} variant={variant}")


@pytest.mark.parametrize("case", ["tile_sk_moe", "tile_moe"])
def test_moe_timeout_path_on_tile_kernels(case):
    # a zero wait budget makes the MoE forms of the tile kernel give up on their weight boxes:
    # they must set the timeout bit, drain the copies in flight (and, in the stream-K form,
    # still pass the CTA barrier of the record combine) and leave the context usable
    if case == "tile_sk_moe":
        Ex, N, K, T, top_k, xps = 288, 3072, 4096, 4, 8, False
        p = synth.moe_problem(Ex, N, K, T, top_k, xps, seed=940, device=DEV)
    else:
        Ex, N, K, T, top_k, xps = 16, 64, 256, 2, 2, False
        p = synth.moe_problem(Ex, N, K, T, top_k, xps, seed=941, device=DEV, fill="all")
    assert nv.describe_plan("moe", Ex, N, K, T, top_k).split()[0] == case
    nv.set_wait_budget_ns(0)
    nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], xps, top_k)
    flags = nv.device_status()
    nv.set_wait_budget_ns(None)
    assert flags & nv.DEV_TIMEOUT
    y = nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], xps, top_k)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]),
                                  synth.bf16_bits(p["x"]), xps, top_k)
    assert bad == 0
    assert_parity(y, yr, ya, f"after timeout ({case})")


def test_moe_many_slots_with_invalid_ids_and_odd_counts():
    # 37 tokens x top-3 = 111 slots (no multiple of 32): some ids out of range (-1, E, E + 7)
    # zero their slots and set DEV_BAD_EXPERT; the others match the oracle
    T, top_k = 37, 3
    N, K = 512, 1024
    ids = synth.routing(T, top_k, E, 940).clone()
    ids[5], ids[40], ids[77], ids[110] = -1, E, E + 7, -1
    p = synth.moe_problem(E, N, K, T, top_k, True, seed=940, device=DEV, ids=ids)
    assert nv.describe_plan("moe_per_slot", E, N, K, T, top_k).split()[0] == "tile_sk_moe"
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], True, top_k, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & nv.DEV_BAD_EXPERT
    assert nv.device_status() & nv.DEV_BAD_EXPERT  # read and cleared here
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]),
                                  synth.bf16_bits(p["x"]), True, top_k)
    assert bad == 4
    assert not torch.any(y[[5, 40, 77, 110]])
    assert_parity(y, yr, ya, "111 slots with invalid ids")


@pytest.mark.parametrize("routing", ["one_expert", "all_distinct"])
def test_moe_256_slots_extreme_routings(routing):
    # every slot on one expert (32 groups of 8) or every slot on its own expert
    T, top_k = 256, 1
    N, K = 256, 512
    ids = torch.full((T,), 17, dtype=torch.int32) if routing == "one_expert" else torch.arange(T, dtype=torch.int32)
    p = synth.moe_problem(E, N, K, T, top_k, True, seed=950, device=DEV, ids=ids)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = nv.moe_gemv(p["w"], p["s"], p["gs"], p["ids"], p["x"], True, top_k, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    yr, ya, bad = oracle.moe_gemv(host(p["w"]), host(p["s"]), host(p["gs"]), host(p["ids"]),
                                  synth.bf16_bits(p["x"]), True, top_k)
    assert bad == 0
    assert_parity(y, yr, ya, f"256 slots, {routing}")
