"""Host replay of the warp-tile kernels' plans and index arithmetic (tests/replay/tile_replay.cu).

The replay includes the library source, runs its planner for a described GB300 on the CPU and
walks every partition and shared-memory index the kernels form (see the file's header). It is
compiled with nvcc to PTX only for the device part: nothing runs on a GPU.
"""
import os
import shutil
import subprocess

import pytest

from nvfp4_weight_only_gemv_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "replay", "tile_replay.cu")


@pytest.mark.parametrize("aligned", [0, 1])
def test_tile_plans_and_indexes(tmp_path, aligned):
    # aligned = 1: the build switch that lets the planner keep stream-K CTAs inside one group
    try:
        nvcc = build.nvcc_path()
    except RuntimeError:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "tile_replay")
    inc = os.path.join(os.path.dirname(HERE), "include")
    cmd = [nvcc, "-O1", "-std=c++17", "-I", inc, "-gencode=arch=compute_103a,code=compute_103a",
           f"-DNVFP4_SK_GROUP_ALIGNED={aligned}", "-o", exe, SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    out = run.stdout.strip().splitlines()
    assert run.returncode == 0 and out and out[-1].endswith("fails 0"), run.stdout[-3000:]
    counts = dict(part.rsplit(" ", 1) for part in out[-1].split(", "))
    assert int(counts["per-item plans"]) >= 300 and int(counts["fused gate/up plans"]) >= 150
    assert int(counts["MoE plans"]) == 5 and int(counts["large MoE plans"]) == 32
    assert (int(counts["group-aligned"]) >= 1) == bool(aligned)
    assert int(counts["FFN plans"]) >= 100 and int(counts["random plans"]) >= 300
