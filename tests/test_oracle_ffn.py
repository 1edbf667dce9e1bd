"""Pins of the oracle's FFN block (CPU only): bf16 rounding of h, then the composition.

The FFN follows the shared-expert nodes of "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json"
(block l3.moe: shared_gate_up, shared_clamp, shared_act, shared_down, one fused group): the
activation h = silu(clamp(gate)) * clamp(up) is stored as bf16 (the silu_mul node's output
precision) and the down projection reads that bf16 h.

- bf16 rounding is pinned by exhaustive round trips of every bf16 value, ties to even at every
  midpoint between neighbours, a library cross-check (PyTorch's float32 -> bfloat16 conversion
  rounds to nearest even, and float32 -> fp64 is exact) and hand values at the edges.
- The composition is pinned by a closed form: a one-hot x and one-hot weights make every gate
  and up value a single E2M1 value times its global scale, so h follows from math.exp, and
  every y from two bf16 h values; plus invariants and exact agreement with the pinned parts.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gemv_gb300 import synth

E2M1 = {0.0: 0x0, 0.5: 0x1, 1.0: 0x2, 1.5: 0x3, 2.0: 0x4, 3.0: 0x5, 4.0: 0x6, 6.0: 0x7}


def _is_nan_bits(b):
    return (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def test_bf16_rne_round_trips_every_bf16_value():
    bits = np.array([b for b in range(1 << 16) if not _is_nan_bits(b)], dtype=np.uint16)
    vals = np.array([oracle.bf16(int(b)) for b in bits])
    assert np.array_equal(oracle.bf16_rne(vals), bits)


def test_bf16_rne_ties_to_even_and_neighbours():
    # positive finite neighbours b, b + 1 (0 .. 0x7F7F): the midpoint is exact in fp64
    lo = np.arange(0, 0x7F7F, dtype=np.int64)
    a = np.array([oracle.bf16(int(b)) for b in lo])
    c = np.array([oracle.bf16(int(b) + 1) for b in lo])
    mid = (a + c) / 2
    even = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(oracle.bf16_rne(mid).astype(np.int64), even)
    assert np.array_equal(oracle.bf16_rne(np.nextafter(mid, np.inf)).astype(np.int64), lo + 1)
    assert np.array_equal(oracle.bf16_rne(np.nextafter(mid, -np.inf)).astype(np.int64), lo)
    # sign symmetry on a sample
    sample = mid[::97]
    assert np.array_equal(oracle.bf16_rne(-sample), oracle.bf16_rne(sample) | 0x8000)


def test_bf16_rne_matches_pytorch_float32_conversion():
    rng = np.random.default_rng(5)
    mant = rng.uniform(1.0, 2.0, 60000)
    expo = rng.integers(-149, 128, 60000)
    v = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)  # some overflow to inf
    v = v * np.where(rng.integers(0, 2, v.size) == 1, 1, -1).astype(np.float32)
    v = np.concatenate([v, rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    v = v[~np.isnan(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(v.astype(np.float64)), ref)


def test_bf16_rne_edges():
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127                  # largest finite bf16, 0x7F7F
    assert oracle.bf16_rne([big])[0] == 0x7F7F
    assert oracle.bf16_rne([(2.0 - 2.0 ** -8) * 2.0 ** 127])[0] == 0x7F80  # tie: to even (inf)
    assert oracle.bf16_rne([np.nextafter((2.0 - 2.0 ** -8) * 2.0 ** 127, 0)])[0] == 0x7F7F
    assert oracle.bf16_rne([2.0 ** -133])[0] == 0x0001          # smallest subnormal
    assert oracle.bf16_rne([2.0 ** -134])[0] == 0x0000          # tie with zero: to even
    assert oracle.bf16_rne([1.5 * 2.0 ** -134])[0] == 0x0001
    assert oracle.bf16_rne([2.0 ** -126])[0] == 0x0080          # smallest normal
    assert oracle.bf16_rne([-0.0])[0] == 0x8000 and oracle.bf16_rne([0.0])[0] == 0x0000
    assert oracle.bf16_rne([math.inf, -math.inf]).tolist() == [0x7F80, 0xFF80]
    assert oracle.bf16_rne([math.nan])[0] == 0x7FC0
    assert oracle.bf16_rne([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]).tolist() == [0x3F80, 0x3F82]


def silu(v):
    return v / (1.0 + math.exp(-v))


def hand_worked_ffn(lib=None):
    """A closed-form FFN: returns (y, y_expected, h_bits, h_bits_expected, h, h_expected).

    H = 32, I = 16, M = 1, x one-hot at k = 0 (1.0). Gate row i holds one E2M1 value a_i at
    k = 0 (scale 1.0), so gate_i = gg * a_i; up likewise. Down row n holds +1.0 at column
    p(n) = (5n + 3) mod 16 and -0.5 at q(n) = (p(n) + 1 + n mod 15) mod 16 (never p(n)), so
    y_n = gd * (h_bits[p(n)] - 0.5 * h_bits[q(n)]) exactly."""
    H, I = 32, 16
    gg, gu, gd, lim = 0.75, 1.25, 0.5, 2.5
    a_vals = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0, 1.0]
    u_vals = [1.0, -1.5, 2.0, 0.5, -3.0, 1.0, 6.0, -1.0, 4.0, 1.5, -6.0, 2.0, 3.0, -0.5, 1.0, -2.0]
    def code(v):
        return E2M1[abs(v)] | (0x8 if v < 0 else 0)
    wg = np.zeros((I, H // 2), dtype=np.uint8)
    wu = np.zeros((I, H // 2), dtype=np.uint8)
    for i in range(I):
        wg[i, 0] = code(a_vals[i])
        wu[i, 0] = code(u_vals[i])
    sgu = np.full((I, H // 16), 0x38, dtype=np.uint8)
    wd = np.zeros((H, I // 2), dtype=np.uint8)
    p = [(5 * n + 3) % 16 for n in range(H)]
    q = [(p[n] + 1 + n % 15) % 16 for n in range(H)]
    for n in range(H):
        wd[n, p[n] // 2] |= code(1.0) << (4 * (p[n] % 2))
        wd[n, q[n] // 2] |= code(-0.5) << (4 * (q[n] % 2))
    sdn = np.full((H, I // 16), 0x38, dtype=np.uint8)
    x = np.zeros((1, H), dtype=np.uint16)
    x[0, 0] = 0x3F80
    y, _, aux = oracle.ffn_swiglu(wg, sgu, gg, wu, sgu, gu, wd, sdn, gd, x, lim, lib=lib)
    clamp = lambda v: min(max(v, -lim), lim)
    h_exp = np.array([silu(clamp(gg * a_vals[i])) * clamp(gu * u_vals[i]) for i in range(I)])
    hb_exp = oracle.bf16_rne(h_exp)  # the rounding is pinned on its own above
    hv = [oracle.bf16(int(b)) for b in hb_exp]
    y_exp = np.array([[gd * (hv[p[n]] - 0.5 * hv[q[n]]) for n in range(H)]])
    return y, y_exp, aux["h_bits"][0], hb_exp, aux["h"][0], h_exp


def test_ffn_hand_worked_closed_form():
    y, y_exp, hb, hb_exp, h, h_exp = hand_worked_ffn()
    assert np.allclose(h, h_exp, rtol=1e-15, atol=0)
    assert np.array_equal(hb, hb_exp)
    assert np.array_equal(y, y_exp)
    # the rounding is visible: some h values are not bf16 numbers
    assert np.any(np.array([oracle.bf16(int(b)) for b in hb]) != h_exp)


def test_ffn_equals_its_pinned_parts():
    p = synth.ffn_problem(64, 48, 3, 7)
    args = [p[k].numpy() if torch.is_tensor(p[k]) else p[k] for k in ("wg", "sg", "gg", "wu", "su", "gu")]
    x = synth.bf16_bits(p["x"])
    y, ya, aux = oracle.ffn_swiglu(*args, p["wd"].numpy(), p["sd"].numpy(), p["gd"], x, 1.5)
    h, hx = oracle.gate_up_swiglu(*args, x, 1.5)
    assert np.array_equal(aux["h"], h)
    for k in ("gate", "gate_abs", "up", "up_abs"):
        assert np.array_equal(aux[k], hx[k])
    hb = oracle.bf16_rne(h)
    assert np.array_equal(aux["h_bits"], hb)
    y2, ya2 = oracle.gemv(p["wd"].numpy(), p["sd"].numpy(), p["gd"], hb)
    assert np.array_equal(y, y2) and np.array_equal(ya, ya2)
    rows = np.array([63, 0, 17], dtype=np.int64)
    y3, _, _ = oracle.ffn_swiglu(*args, p["wd"].numpy(), p["sd"].numpy(), p["gd"], x, 1.5, rows=rows)
    assert np.array_equal(y3, y[:, rows])


def test_ffn_invariants():
    p = synth.ffn_problem(48, 32, 2, 9)
    args = [p[k].numpy() if torch.is_tensor(p[k]) else p[k] for k in ("wg", "sg", "gg", "wu", "su", "gu")]
    wd, sd = p["wd"].numpy(), p["sd"].numpy()
    x = synth.bf16_bits(p["x"])
    y, ya, aux = oracle.ffn_swiglu(*args, wd, sd, p["gd"], x)
    # zero x: gate = up = 0, h = 0, y = 0
    y0, _, a0 = oracle.ffn_swiglu(*args, wd, sd, p["gd"], np.zeros_like(x))
    assert not np.any(y0) and not np.any(a0["h_bits"] & 0x7FFF)
    # a power of two on the down scale scales y exactly
    y2, _, _ = oracle.ffn_swiglu(*args, wd, sd, 4.0 * p["gd"], x)
    assert np.array_equal(y2, 4.0 * y)
    # permuting the down rows permutes y
    perm = np.random.default_rng(1).permutation(48)
    yp, _, _ = oracle.ffn_swiglu(*args, wd[perm], sd[perm], p["gd"], x)
    assert np.array_equal(yp, y[:, perm])
    # rounding h moves y by at most half a bf16 ulp of every h term: |dy| <= 2^-8 * yabs
    E = np.array([oracle.e2m1(c) for c in range(16)])
    dq = np.repeat(np.array([[oracle.e4m3(int(c)) for c in row] for row in sd]), 16, axis=1)
    wv = np.stack([E[wd & 15], E[wd >> 4]], axis=-1).reshape(48, 32) * dq
    y_unrounded = p["gd"] * (aux["h"] @ wv.T)
    assert np.all(np.abs(y - y_unrounded) <= 2.0 ** -8 * ya)
    assert np.any(y != y_unrounded)


def test_ffn_rejects_bad_arguments():
    w = np.zeros((16, 8), np.uint8)
    s = np.zeros((16, 1), np.uint8)
    with pytest.raises(ValueError):
        oracle.ffn_swiglu(w, s, 1.0, w, s, 1.0, w, s, 1.0, np.zeros((1, 16), np.uint16), lim=0.0)
