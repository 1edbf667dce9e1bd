"""Pins of the oracle's scale-dictionary GEMV (CPU only).

The dictionary form changes only where a block's scale code comes from: code = dict[index].
So it is pinned by (1) hand-worked examples of the index layout (tests/golden/
sdict_hand_worked.json, typed by hand from their derivations), (2) an independent bit reader
in this file against the oracle's index extraction at every position, and (3) exact equality
with the plain oracle (itself pinned in test_oracle_pins.py) on the same weights with the
scale codes dict[index] written out, dense and routed-expert. The index layout is this
project's reading of "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[64] (4.3125
bit/weight with a scale dictionary): see the comment above nvfp4_oracle_sdict_index.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gemv_gb300 import synth

from conftest import GOLDEN


def pack_indices(ind: np.ndarray, N: int, K: int) -> np.ndarray:
    """Writes ind [N, K/16] (values 0..31) into the index plane, one bit at a time."""
    segs, tiles = K // 256, (N + 15) // 16
    out = np.zeros(tiles * segs * 160, dtype=np.uint8)
    for n in range(N):
        r, i = divmod(n, 16)
        for b in range(K // 16):
            c, j = divmod(b, 16)
            first = (r * segs + c) * 160 * 8 + 5 * (16 * i + j)  # bit position in the plane
            for t in range(5):
                if (int(ind[n, b]) >> t) & 1:
                    out[(first + t) // 8] |= np.uint8(1 << ((first + t) % 8))
    return out


def read_index(plane: np.ndarray, K: int, n: int, b: int) -> int:
    """The index of block b of row n, read as a slice of the record's little-endian integer."""
    r, i = divmod(n, 16)
    c, j = divmod(b, 16)
    rec = int.from_bytes(plane[(r * (K // 256) + c) * 160:(r * (K // 256) + c + 1) * 160].tobytes(), "little")
    return (rec >> (5 * (16 * i + j))) & 31


def random_case(N, K, M, seed):
    rng = np.random.default_rng(seed)
    w = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    sdict = rng.choice(codes, 32, replace=False).astype(np.uint8)
    ind = rng.integers(0, 32, (N, K // 16))
    x = synth.bf16_bits(synth.random_x(M, K, seed))
    return w, sdict, ind, x


def _golden():
    return json.load(open(os.path.join(GOLDEN, "sdict_hand_worked.json")))


@pytest.mark.parametrize("ex", _golden()["examples"], ids=lambda e: e["name"])
def test_hand_worked_examples(ex):
    N, K = ex["N"], ex["K"]
    w = np.frombuffer(bytes.fromhex(ex["w_row"]) * N, dtype=np.uint8).reshape(N, K // 2)
    idx = np.frombuffer(bytes.fromhex(ex["idx"]), dtype=np.uint8)
    assert idx.size == oracle.sdict_idx_bytes(N, K)
    sdict = np.array([int(v, 16) for v in ex["dict"]], dtype=np.uint8)
    x = np.full((ex["M"], K), int(ex["x_value"], 16), dtype=np.uint16)
    y, _ = oracle.gemv_sdict(w, idx, sdict, ex["g"], x)
    assert np.array_equal(y, np.array([ex["y"]]))


@pytest.mark.parametrize("N,K", [(16, 256), (40, 512), (33, 768), (1, 256)])
def test_index_extraction_matches_an_independent_reader(N, K):
    _, _, ind, _ = random_case(N, K, 1, 7 + N)
    plane = pack_indices(ind, N, K)
    assert plane.size == oracle.sdict_idx_bytes(N, K) == ((N + 15) // 16) * (K // 256) * 160
    for n in range(N):
        for b in range(K // 16):
            assert read_index(plane, K, n, b) == ind[n, b]
            assert oracle.sdict_index(plane, K, n, b) == ind[n, b]


@pytest.mark.parametrize("N,K", [(16, 256), (40, 512), (33, 768), (1, 256), (130, 4096)])
def test_generator_packer_matches_the_bitwise_one(N, K):
    # the input generator's vectorised packer (which GPU tests and the benchmark use) writes
    # the same bytes as this file's bit-by-bit packer
    _, _, ind, _ = random_case(N, K, 1, 3 + N)
    assert np.array_equal(synth.sdict_pack(torch.from_numpy(ind), N, K).numpy(), pack_indices(ind, N, K))


def test_generator_dictionary_form_round_trips():
    w, s, g = synth.random_weight_sdict(300, 1024, 5, max_codes=12)
    plane, table = synth.sdict_form(s)
    codes = np.unique(s.numpy())
    assert codes.size <= 12 and np.array_equal(table.numpy()[:codes.size], codes)
    for n in (0, 17, 299):
        for b in (0, 5, 63):
            assert table[oracle.sdict_index(plane.numpy(), 1024, n, b)] == s[n, b]


@pytest.mark.parametrize("N,K,M", [(16, 256, 1), (40, 512, 3), (77, 1024, 2), (5, 256, 8)])
def test_equals_plain_oracle_with_the_codes_written_out(N, K, M):
    # 5-bit indices that reach every table entry, NaN-free random codes and E2M1 bytes
    w, sdict, ind, x = random_case(N, K, M, 100 + N)
    plane = pack_indices(ind, N, K)
    s = sdict[ind].astype(np.uint8)
    y_d, ya_d = oracle.gemv_sdict(w, plane, sdict, 0.375, x)
    y_p, ya_p = oracle.gemv(w, s, 0.375, x)
    assert np.array_equal(y_d, y_p) and np.array_equal(ya_d, ya_p)
    rows = np.array([N - 1, 0, N // 2], dtype=np.int64)
    y_r, _ = oracle.gemv_sdict(w, plane, sdict, 0.375, x, rows=rows)
    assert np.array_equal(y_r, y_p[:, rows])


def test_a_nan_table_entry_poisons_only_its_blocks_rows():
    N, K, M = 32, 256, 1
    w, sdict, ind, x = random_case(N, K, M, 5)
    sdict = sdict.copy()
    sdict[3] = 0x7F
    ind = np.zeros_like(ind)
    ind[9, 4] = 3
    y, _ = oracle.gemv_sdict(w, pack_indices(ind, N, K), sdict, 1.0, x)
    assert np.isnan(y[0, 9]) and np.isfinite(np.delete(y[0], 9)).all()


@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_equals_plain_moe_oracle(x_per_slot):
    E, N, K, T, top_k = 5, 24, 512, 3, 2
    rng = np.random.default_rng(11)
    w = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    sdict = np.stack([rng.choice(codes, 32, replace=False) for _ in range(E)]).astype(np.uint8)
    ind = rng.integers(0, 32, (E, N, K // 16))
    planes = np.stack([pack_indices(ind[e], N, K) for e in range(E)])
    s = np.stack([sdict[e][ind[e]] for e in range(E)]).astype(np.uint8)
    gs = rng.uniform(0.5, 2.0, E).astype(np.float32)
    ids = np.array([4, 0, 2, 2, 1, 4], dtype=np.int32)
    x = synth.bf16_bits(synth.random_x(T * top_k if x_per_slot else T, K, 12))
    y_d, ya_d, bad_d = oracle.moe_gemv_sdict(w, planes, sdict, gs, ids, x, x_per_slot, top_k)
    y_p, ya_p, bad_p = oracle.moe_gemv(w, s, gs, ids, x, x_per_slot, top_k)
    assert bad_d == bad_p == 0
    assert np.array_equal(y_d, y_p) and np.array_equal(ya_d, ya_p)
    # an out-of-range id zeroes its slot in both forms
    ids2 = ids.copy()
    ids2[3] = 9
    y_d, _, bad_d = oracle.moe_gemv_sdict(w, planes, sdict, gs, ids2, x, x_per_slot, top_k)
    assert bad_d == 1 and np.all(y_d[3] == 0)


def test_rejects_k_not_multiple_of_256():
    w = np.zeros((16, 64), dtype=np.uint8)
    with pytest.raises((ValueError, AssertionError)):
        oracle.gemv_sdict(w, np.zeros(0, np.uint8), np.zeros(32, np.uint8), 1.0, np.zeros((1, 128), np.uint16))
