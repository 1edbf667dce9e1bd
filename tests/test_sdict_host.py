"""The scale-dictionary format on the host (no GPU): the library's encoder writes the index plane
and table that an independent bit packer (test_oracle_sdict.pack_indices) writes, rejects
tensors with more than 32 codes, and the C ABI validates the dictionary entry points before it
touches the CUDA runtime; the planner gives the workload shapes the tile kernels' dictionary
forms."""
import ctypes

import numpy as np
import pytest
import torch

import nvfp4_weight_only_gemv_gb300 as nv
from nvfp4_weight_only_gemv_gb300 import synth

from test_oracle_sdict import pack_indices
from test_plans_host import fits, plan


@pytest.mark.parametrize("N,K,ncodes", [(16, 256, 32), (40, 512, 7), (33, 768, 1), (300, 4096, 20), (0, 256, 0)])
def test_encoder_matches_an_independent_packer(N, K, ncodes):
    rng = np.random.default_rng(N + K)
    codes = np.sort(rng.choice(np.array([c for c in range(256) if c not in (0x7F, 0xFF)]), ncodes, replace=False))
    ind = rng.integers(0, max(ncodes, 1), (N, K // 16))
    if N and ncodes:
        ind.reshape(-1)[:ncodes] = np.arange(ncodes)  # every code is used
    s = torch.from_numpy(codes[ind].astype(np.uint8) if ncodes else np.zeros((N, K // 16), np.uint8))
    plane, table = nv.sdict_encode(s)
    assert plane.numel() == nv.sdict_plane_bytes(N, K) == ((N + 15) // 16) * (K // 256) * 160
    if ncodes:
        # codes in increasing byte order, the rest of the table repeats the last one
        assert np.array_equal(table.numpy()[:ncodes], codes)
        assert np.all(table.numpy()[ncodes:] == codes[-1])
        assert np.array_equal(plane.numpy(), pack_indices(ind, N, K))


def test_encoder_per_expert_and_more_than_32_codes():
    p = synth.moe_problem(3, 32, 512, 2, 2, False, seed=5, fill="all")
    s = p["s"]
    if max(len(np.unique(s[e].numpy())) for e in range(3)) <= 32:
        planes, tables = nv.sdict_encode(s)
        assert planes.shape == (3, nv.sdict_plane_bytes(32, 512)) and tables.shape == (3, 32)
    wide = torch.arange(64, dtype=torch.uint8).repeat(16, 1)   # [16, 64]: 64 distinct codes, K = 1024
    assert len(np.unique(wide.numpy())) > 32
    with pytest.raises(ValueError):
        nv.sdict_encode(wide)
    with pytest.raises(ValueError):
        nv.sdict_plane_bytes(16, 272)


P = ctypes.c_void_p
FAKE = P(4096)  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("args,expect", [
    ((None, FAKE, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 256, None), 1),      # null weights
    ((FAKE, None, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 256, None), 1),      # null index plane
    ((FAKE, FAKE, None, 1.0, FAKE, FAKE, 0, 1, 16, 256, None), 1),      # null table
    ((FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, 0, 9, 16, 256, None), 2),      # M > 8
    ((FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, 0, 1, 16, 272, None), 2),      # K % 256 != 0
    ((FAKE, FAKE, FAKE, 1.0, FAKE, FAKE, 5, 1, 16, 256, None), 4),      # bad output type
])
def test_dense_sdict_validation(args, expect):
    assert nv.library().nvfp4_gemv_sdict(*args) == expect


def test_moe_sdict_validation():
    lib = nv.library()
    base = [FAKE, FAKE, FAKE, FAKE, 8, FAKE, 2, 2, FAKE, 0, FAKE, 0, 64, 256, None, None]
    assert lib.nvfp4_moe_gemv_sdict(*base[:2], None, *base[3:]) == 1
    bad_k = list(base)
    bad_k[13] = 272
    assert lib.nvfp4_moe_gemv_sdict(*bad_k) == 2
    bad_e = list(base)
    bad_e[4] = 0
    assert lib.nvfp4_moe_gemv_sdict(*bad_e) == 2


@pytest.mark.parametrize("kind,M,N,K,T,top_k", [
    ("dense_sdict", 1, 4096, 4096, 0, 0), ("dense_sdict", 5, 1024, 4096, 0, 0),
    ("dense_sdict", 1, 151936, 4096, 0, 0), ("dense_sdict", 8, 4096, 12288, 0, 0),
    ("moe_sdict", 288, 3072, 4096, 4, 8), ("moe_per_slot_sdict", 288, 4096, 1536, 4, 8)])
def test_workload_shapes_take_the_dictionary_tile_kernels(kind, M, N, K, T, top_k):
    name, f = plan(kind, M, N, K, T, top_k)
    assert name == ("tile_sdict" if kind == "dense_sdict" else "tile_sk_moe_sdict")
    assert fits(f)
    if kind != "dense_sdict":
        assert f["group_aligned"] == 1


def test_dictionary_fallbacks():
    assert plan("dense_sdict", 1, 100, 528)[0] == "simple"                 # K % 256 != 0
    assert plan("moe_sdict", 288, 3072, 4096, 32, 8)[0] == "tile_sk_moe_sdict"  # 256 slots, one group per CTA
    assert plan("moe_sdict", 40, 512, 1024, 100, 3)[0] == "simple"         # > 256 slots
