"""The FFN block's entry point without a caller workspace (nvfp4_ffn_swiglu_static).

It runs the same kernels as nvfp4_ffn_swiglu with the library's own 256 KB device array as the
workspace. Two calls in a row on the same inputs must give bitwise the same y as the entry point
with a caller workspace (the kernels and plans are the same and deterministic), on a shape that
runs as one launch and one that runs as two; a size beyond the array is rejected. This file is
collected last, so it also runs after every other GPU test has used the library.
"""
import pytest
import torch

import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _args(H, I, M, seed):
    p = synth.ffn_problem(H, I, M, seed, device=DEV)
    w = [p[k] for k in ("wg", "sg", "gg", "wu", "su", "gu", "wd", "sd", "gd")]
    return w, p["x"]


@pytest.mark.parametrize("H,I,M,out", [(4096, 768, 2, torch.bfloat16), (4096, 12288, 1, torch.float32)])
def test_static_workspace_matches_caller_workspace_twice(H, I, M, out):
    w, x = _args(H, I, M, 900 + M)
    ws = nv.ffn_workspace(M, I)
    for call in range(2):
        x_c = x if call == 0 else synth.random_x(M, H, 950 + call, device=DEV)
        ref = nv.ffn_swiglu(*w, x_c, 10.0, workspace=ws, out_dtype=out)
        got = nv.ffn_swiglu_static(*w, x_c, 10.0, out_dtype=out)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}: {int((got != ref).sum())} outputs differ"
    assert nv.device_status() == 0


def test_static_workspace_rejects_sizes_beyond_its_array():
    w, x = _args(256, 256, 1, 960)
    # M * I beyond 130048: nvfp4_ffn_workspace_bytes(8, 16384) = 2048 + 262144 > 262144
    e = torch.zeros(16384, 128, dtype=torch.uint8, device=DEV)
    es = torch.zeros(16384, 16, dtype=torch.uint8, device=DEV)
    d = torch.zeros(256, 8192, dtype=torch.uint8, device=DEV)
    ds = torch.zeros(256, 1024, dtype=torch.uint8, device=DEV)
    x8 = torch.zeros(8, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.ffn_swiglu_static(e, es, 1.0, e, es, 1.0, d, ds, 1.0, x8, 1.0)
    assert ei.value.status == 5  # NVFP4_ERR_UNSUPPORTED
