"""The launch planner, run on the host for a described GB300 (152 SMs, 227 KB of shared memory
a CTA may opt into, 228 KB per SM): no GPU needed. Checks which kernel each call shape gets
and that every plan fits the device."""
import re

import pytest

import nvfp4_weight_only_gemv_gb300 as nv

SMS, OPTIN, PER_SM = 152, 232448, 233472


def plan(kind, M, N, K, T=0, top_k=0, **dev):
    desc = nv.describe_plan_host(kind, M, N, K, T, top_k, **dev)
    name = desc.split()[0]
    fields = {k: int(v) for k, v in re.findall(r"(\w+)=(\d+)", desc)}
    return name, fields


def fits(f, sms=SMS, optin=OPTIN, per_sm=PER_SM):
    if f["smem"] > optin:
        return False
    # a grid above one CTA per SM needs two CTAs' shared memory on an SM (1 KB reserved each)
    if f["grid"] > sms and 2 * (f["smem"] + 1024) > per_sm:
        return False
    return f["grid"] % f["split"] == 0


@pytest.mark.parametrize("kind,M,N,K", [
    ("dense", 1, 4096, 4096), ("dense", 5, 4096, 4096), ("dense", 1, 1024, 4096), ("dense", 5, 1024, 4096),
    ("gate_up", 1, 12288, 4096), ("gate_up", 8, 12288, 4096), ("dense", 1, 4096, 12288),
    ("dense", 8, 4096, 12288), ("dense", 1, 151936, 4096), ("gate_up_swiglu", 1, 12288, 4096),
    ("gate_up_swiglu", 8, 12288, 4096), ("dense", 1, 256, 512)])
def test_workload_shapes_take_the_tile_kernel(kind, M, N, K):
    name, f = plan(kind, M, N, K)
    assert name == ("tile_swiglu" if kind == "gate_up_swiglu" else "tile")
    assert f["block"] == 256 and fits(f)
    assert f["rows_per_item"] * f["k_warps"] == 128          # 8 warps: tiles per item x K split
    assert 2 <= f["stages"] <= 4


def test_large_problems_fill_every_sm_twice():
    for kind, M, N, K in (("dense", 1, 151936, 4096), ("gate_up", 1, 12288, 4096)):
        _, f = plan(kind, M, N, K)
        assert f["grid"] == 2 * SMS


def test_fused_swiglu_items_hold_whole_gate_up_pairs():
    for M in range(1, 9):
        for N, K in ((12288, 4096), (37, 2560), (1000, 1024), (4096, 1536), (1, 256)):
            name, f = plan("gate_up_swiglu", M, N, K)
            assert name == "tile_swiglu" and fits(f)
            assert (f["rows_per_item"] // 16) % 2 == 0 and f["k_warps"] <= 4


@pytest.mark.parametrize("kind,T,N,K", [("moe", 4, 3072, 4096), ("moe_per_slot", 4, 4096, 1536)])
def test_routed_experts_take_the_stream_k_form(kind, T, N, K):
    name, f = plan(kind, 288, N, K, T, 8)
    assert name == "tile_sk_moe" and fits(f)
    assert f["grid"] == 2 * SMS


def test_fallback_kernels():
    assert plan("moe", 288, 3072, 4064, 8, 8)[0] == "stream_moe"      # K % 256 != 0, K % 32 == 0
    assert plan("moe", 40, 64, 256, 100, 3)[0] == "simple"            # 300 slots: above every tiled limit
    assert plan("dense", 1, 100, 4064)[0] == "stream"                  # K % 256 != 0, K % 32 == 0
    assert plan("dense", 1, 100, 528)[0] == "simple"                   # K % 32 != 0
    assert plan("gate_up_swiglu", 1, 100, 4064)[0] == "simple"         # no streaming form fused
    for kind in ("dense", "gate_up"):
        name, f = plan(kind, 3, 1000, 4064)
        assert name == "stream" and fits(f)


def test_other_device_descriptions():
    # a device with fewer SMs and a smaller shared memory: plans shrink to fit it
    dev = dict(sm_count=100, smem_optin=101376, smem_per_sm=102400)
    for kind, M, N, K in (("dense", 1, 4096, 4096), ("dense", 8, 4096, 12288), ("gate_up_swiglu", 4, 12288, 4096)):
        name, f = plan(kind, M, N, K, **dev)
        assert fits(f, 100, 101376, 102400), (kind, M, N, K, f)


def test_bad_descriptions_are_rejected():
    with pytest.raises(ValueError):
        nv.describe_plan_host("dense", 1, 256, 512, sm_count=0)
    with pytest.raises(ValueError):
        nv.describe_plan_host("dense", 1, 256, 512, smem_optin=4096, smem_per_sm=1024)


@pytest.mark.parametrize("value,kernel", [("3", "stream"), ("1", "simple"), ("0", "tile"), ("7", "tile"),
                                          ("x", "tile")])
def test_force_variant_environment(value, kernel):
    # NVFP4_GEMV_FORCE_VARIANT sets the library's starting kernel selection (0..3, else ignored)
    import subprocess
    import sys
    code = ("import nvfp4_weight_only_gemv_gb300 as nv; "
            "print(nv.describe_plan_host('dense', 1, 4096, 4096).split()[0])")
    env = dict(__import__("os").environ, NVFP4_GEMV_FORCE_VARIANT=value)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == kernel


@pytest.mark.parametrize("x_per_slot,N,K", [(False, 3072, 4096), (True, 4096, 1536)])
@pytest.mark.parametrize("T", [5, 8, 16, 32])
def test_larger_moe_routings_take_the_stream_k_form(x_per_slot, N, K, T):
    # 40..256 slots: the stream-K tile kernel (groups built by the whole CTA, a window of up
    # to 4 of them per CTA), no longer the streaming kernel
    name, f = plan("moe_per_slot" if x_per_slot else "moe", 288, N, K, T, 8)
    assert name == "tile_sk_moe" and fits(f) and f["mt"] == 8
