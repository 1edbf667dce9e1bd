"""Pins for the CPU oracle. It is checked against things other than itself.

* Golden fixtures: the E2M1 value set, E4M3 spot values, and hand-worked examples.
* torch's float8_e4m3fn and bf16 decoders (library routines) over every code.
* Closed forms and invariants: zero input, one-hot x, linearity in the global
  scale, permutation of K-blocks, gate/up concatenation, MoE with one expert.
* numpy float64 matmul of an independently dequantised weight.
* Exact rational arithmetic (fractions.Fraction) on tiny inputs.

The test-side dequantiser below uses the golden E2M1 table and torch's E4M3
decoder. It shares no code with the oracle.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gemv_gb300 import synth

from conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


E2M1_TABLE = np.array([_golden("e2m1_values.json")["values"][str(c)] for c in range(16)],
                      dtype=np.float64)


def torch_e4m3(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_bf16(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def dequant(w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Independent dequantiser: [N, K/2] codes + [N, K/16] scales -> fp64 [N, K]."""
    lo = w & 0xF
    hi = w >> 4
    codes = np.empty((w.shape[0], w.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    scale = np.repeat(torch_e4m3(s), 16, axis=1)
    return E2M1_TABLE[codes] * scale


def _arrays(ex):
    w = np.array([list(bytes.fromhex(r)) for r in ex["w"]], dtype=np.uint8)
    s = np.array([list(bytes.fromhex(r)) for r in ex["s"]], dtype=np.uint8)
    x = np.array([[int(h, 16) for h in row] for row in ex["x"]], dtype=np.uint16)
    return w, s, x


def _rand_problem(N, K, M, seed):
    p = synth.dense_problem(N, K, M, seed)
    return p["w"].numpy(), p["s"].numpy(), p["g"], synth.bf16_bits(p["x"])


# ---------------------------------------------------------------- decoders

def test_e2m1_matches_value_set():
    for c in range(16):
        got = oracle.e2m1(c)
        assert got == E2M1_TABLE[c], c
        assert math.copysign(1.0, got) == math.copysign(1.0, E2M1_TABLE[c]), c


def test_e4m3_all_codes_match_torch():
    ref = torch_e4m3(np.arange(256))
    for c in range(256):
        got = oracle.e4m3(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c], hex(c)
            assert math.copysign(1.0, got) == math.copysign(1.0, ref[c]), hex(c)


def test_e4m3_spot_values():
    g = _golden("e4m3_spot_values.json")
    for h, v in g["values_hex"].items():
        assert oracle.e4m3(int(h, 16)) == v, h
    for h in g["nan_hex"]:
        assert math.isnan(oracle.e4m3(int(h, 16))), h


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # skip inf/NaN patterns
    ref = torch_bf16(bits)
    got = np.array([oracle.bf16(int(b)) for b in bits])
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- hand-worked examples

@pytest.mark.parametrize("idx", range(len(_golden("hand_worked.json")["examples"])))
def test_hand_worked_example(idx):
    ex = _golden("hand_worked.json")["examples"][idx]
    w, s, x = _arrays(ex)
    assert w.shape == (ex["N"], ex["K"] // 2) and x.shape == (ex["M"], ex["K"])
    y, ya = oracle.gemv(w, s, ex["g"], x)
    assert np.array_equal(y, np.array(ex["y"], dtype=np.float64)), ex["name"]
    assert np.all(ya >= np.abs(y))


# ---------------------------------------------------------------- invariants

def test_zero_x_and_zero_weight():
    w, s, g, x = _rand_problem(40, 96, 3, 11)
    y, ya = oracle.gemv(w, s, g, np.zeros_like(x))
    assert np.all(y == 0) and np.all(ya == 0)
    y, _ = oracle.gemv(np.zeros_like(w), s, g, x)
    assert np.all(y == 0)


def test_one_hot_x_selects_one_term():
    w, s, g, x = _rand_problem(24, 64, 1, 12)
    deq = dequant(w, s)
    one = np.uint16(0x3F80)
    for k in (0, 1, 15, 16, 17, 63):
        xk = np.zeros((1, 64), dtype=np.uint16)
        xk[0, k] = one
        y, _ = oracle.gemv(w, s, g, xk)
        assert np.array_equal(y[0], g * deq[:, k]), k


@pytest.mark.parametrize("a", [-3, -1, 1, 4])
def test_linear_in_global_scale(a):
    w, s, g, x = _rand_problem(33, 128, 2, 13)
    y1, _ = oracle.gemv(w, s, g, x)
    y2, _ = oracle.gemv(w, s, g * 2.0 ** a, x)
    assert np.array_equal(y2, y1 * 2.0 ** a)


def test_k_block_permutation_invariance():
    N, K, M = 17, 160, 2
    w, s, g, x = _rand_problem(N, K, M, 14)
    perm = np.random.default_rng(1).permutation(K // 16)
    wp = w.reshape(N, K // 16, 8)[:, perm].reshape(N, K // 2)
    sp = s[:, perm]
    xp = x.reshape(M, K // 16, 16)[:, perm].reshape(M, K)
    y1, ya = oracle.gemv(w, s, g, x)
    y2, _ = oracle.gemv(wp, sp, g, xp)
    assert np.all(np.abs(y1 - y2) <= 1e-13 * ya + 1e-300)


def test_matches_numpy_matmul_of_dequantised_weight():
    N, K, M = 96, 512, 3
    w, s, g, x = _rand_problem(N, K, M, 15)
    ref = g * (torch_bf16(x) @ dequant(w, s).T)
    y, ya = oracle.gemv(w, s, g, x)
    assert np.all(np.abs(y - ref) <= 1e-12 * ya)
    assert np.all(ya >= np.abs(y))
    ref_abs = abs(g) * (np.abs(torch_bf16(x)) @ np.abs(dequant(w, s)).T)
    assert np.allclose(ya, ref_abs, rtol=1e-12, atol=0)


def test_row_subset_matches_full():
    w, s, g, x = _rand_problem(50, 64, 2, 16)
    y, ya = oracle.gemv(w, s, g, x)
    rows = [49, 0, 7, 7, 23]
    ys, yas = oracle.gemv(w, s, g, x, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(yas, ya[:, rows])


def test_nan_scale_propagates_to_its_row_only():
    w, s, g, x = _rand_problem(8, 64, 2, 17)
    s = s.copy()
    s[3, 2] = 0x7F
    y, _ = oracle.gemv(w, s, g, x)
    assert np.all(np.isnan(y[:, 3]))
    assert np.all(np.isfinite(np.delete(y, 3, axis=1)))


def test_sign_bit_scale_negates():
    w, s, g, x = _rand_problem(6, 32, 1, 18)
    y, _ = oracle.gemv(w, s, g, x)
    y2, _ = oracle.gemv(w, s | 0x80, g, x)
    assert np.array_equal(y2, -y)


# ---------------------------------------------------------------- exact arithmetic

def _exact(w, s, g, x):
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    e2 = [Fraction(v) for v in E2M1_TABLE]
    sc = torch_e4m3(s)
    xv = torch_bf16(x)
    out = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                code = (int(w[n, k // 2]) >> (4 * (k % 2))) & 0xF
                acc += e2[code] * Fraction(sc[n, k // 16]) * Fraction(xv[m, k])
            out[m, n] = float(Fraction(g) * acc)
    return out


@pytest.mark.parametrize("N,K,M,seed", [(3, 16, 1, 21), (5, 32, 2, 22), (32, 32, 2, 23)])
def test_fraction_bruteforce_tiny(N, K, M, seed):
    w, s, g, x = _rand_problem(N, K, M, seed)
    # keep |x| in [2^-8, 2^4) so every fp64 partial sum is exact (terms have <= 14
    # significant bits over a limited exponent span); then only g * sum rounds once.
    xv = torch_bf16(x)
    keep = (np.abs(xv) >= 2.0 ** -8) & (np.abs(xv) < 16)
    x = np.where(keep, x, np.uint16(0x3F80)).astype(np.uint16)
    exact = _exact(w, s, g, x)
    y, _ = oracle.gemv(w, s, g, x)
    assert np.array_equal(y, exact)


# ---------------------------------------------------------------- gate/up and MoE

def test_gate_up_is_two_gemvs_side_by_side():
    p = synth.gate_up_problem(40, 96, 3, 31)
    wg, sg, wu, su = (p[k].numpy() for k in ("wg", "sg", "wu", "su"))
    x = synth.bf16_bits(p["x"])
    y, ya = oracle.gemv_gate_up(wg, sg, p["gg"], wu, su, p["gu"], x)
    xv = torch_bf16(x)
    ref = np.concatenate([p["gg"] * (xv @ dequant(wg, sg).T), p["gu"] * (xv @ dequant(wu, su).T)], 1)
    assert y.shape == (3, 80)
    assert np.all(np.abs(y - ref) <= 1e-12 * ya)
    rows = [79, 0, 40, 39]
    ys, _ = oracle.gemv_gate_up(wg, sg, p["gg"], wu, su, p["gu"], x, rows=rows)
    assert np.array_equal(ys, y[:, rows])


@pytest.mark.parametrize("x_per_slot", [False, True])
def test_moe_matches_per_slot_matmul(x_per_slot):
    E, N, K, T, top_k = 12, 24, 64, 3, 4
    p = synth.moe_problem(E, N, K, T, top_k, x_per_slot, seed=41)
    w, s, gs, ids = p["w"].numpy(), p["s"].numpy(), p["gs"].numpy(), p["ids"].numpy()
    x = synth.bf16_bits(p["x"])
    y, ya, bad = oracle.moe_gemv(w, s, gs, ids, x, x_per_slot, top_k)
    assert bad == 0 and y.shape == (T * top_k, N)
    xv = torch_bf16(x)
    for sl in range(T * top_k):
        e = ids[sl]
        xr = xv[sl if x_per_slot else sl // top_k]
        ref = float(gs[e]) * (dequant(w[e], s[e]) @ xr)
        assert np.all(np.abs(y[sl] - ref) <= 1e-12 * ya[sl]), sl


def test_moe_single_expert_reduces_to_dense():
    E, N, K, T, top_k = 5, 16, 48, 2, 3
    p = synth.moe_problem(E, N, K, T, top_k, False, seed=42, fill="all")
    w, s, gs = p["w"].numpy(), p["s"].numpy(), p["gs"].numpy()
    x = synth.bf16_bits(p["x"])
    ids = np.full(T * top_k, 3, dtype=np.int32)
    y, _, _ = oracle.moe_gemv(w, s, gs, ids, x, False, top_k)
    yd, _ = oracle.gemv(w[3], s[3], float(gs[3]), x)
    for sl in range(T * top_k):
        assert np.array_equal(y[sl], yd[sl // top_k])


def test_moe_out_of_range_ids_give_zero_rows():
    E, N, K, T, top_k = 4, 8, 32, 2, 2
    p = synth.moe_problem(E, N, K, T, top_k, True, seed=43, fill="all")
    ids = np.array([0, -1, 4, 3], dtype=np.int32)
    y, ya, bad = oracle.moe_gemv(p["w"].numpy(), p["s"].numpy(), p["gs"].numpy(), ids,
                                 synth.bf16_bits(p["x"]), True, top_k)
    assert bad == 2
    assert np.all(y[1] == 0) and np.all(y[2] == 0)
    assert np.any(y[0] != 0) and np.any(y[3] != 0)


# ---------------------------------------------------------------- fused gate/up activation
# The swiglu_clamp and silu_mul nodes after the gate/up projection ("glm-5.3-flash-nvfp4-
# tp3-512k--gb10 graph.json", block l0.mlp): silu(c(gate)) * c(up), c a clamp whose limit the
# pages do not give (an argument here; +inf for none).

LN3 = math.log(3.0)


def test_silu_closed_forms():
    # the logistic function is exactly 3/4 at ln 3 (exp(-ln 3) = 1/3) and 1/4 at -ln 3
    assert oracle.swiglu(LN3, 1.0) == pytest.approx(0.75 * LN3, rel=1e-15)
    assert oracle.swiglu(-LN3, 1.0) == pytest.approx(-0.25 * LN3, rel=1e-15)
    assert oracle.swiglu(math.log(1.0 / 7.0), 2.0) == pytest.approx(2.0 * math.log(1.0 / 7.0) / 8.0, rel=1e-15)
    assert oracle.swiglu(0.0, 5.0) == 0.0
    # silu(v) tends to v for large v and to 0 for very negative v; its slope at 0 is 1/2
    assert oracle.swiglu(40.0, 1.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(oracle.swiglu(-40.0, 1.0)) < 1e-15
    assert oracle.swiglu(1e-6, 1.0) / 1e-6 == pytest.approx(0.5, rel=1e-5)


def test_silu_odd_part_and_linearity_in_up():
    rng = np.random.default_rng(5)
    for v in rng.normal(0, 3, 40):
        # silu(v) - silu(-v) = v (the logistic function satisfies s(v) + s(-v) = 1)
        assert oracle.swiglu(v, 1.0) - oracle.swiglu(-v, 1.0) == pytest.approx(v, rel=1e-13, abs=1e-15)
        u = rng.normal()
        assert oracle.swiglu(v, 4.0 * u) == 4.0 * oracle.swiglu(v, u)  # power of two: exact


def test_swiglu_clamp_saturates_both_inputs():
    lim = 2.0
    assert oracle.swiglu(5.0, 1.0, lim) == oracle.swiglu(2.0, 1.0)
    assert oracle.swiglu(-5.0, 1.0, lim) == oracle.swiglu(-2.0, 1.0)
    assert oracle.swiglu(1.0, 7.0, lim) == oracle.swiglu(1.0, 2.0)
    assert oracle.swiglu(1.0, -9.0, lim) == oracle.swiglu(1.0, -2.0)
    assert oracle.swiglu(1.5, -1.25, lim) == oracle.swiglu(1.5, -1.25)  # inside: untouched
    assert math.isnan(oracle.swiglu(float("nan"), 1.0, lim))
    assert math.isnan(oracle.swiglu(1.0, float("nan"), lim))


def test_gate_up_swiglu_hand_worked():
    # every code 1.0 (nibble 0x2) with scale 1.0 (0x38), K = 16 and x = 1: each dot product is
    # 16, so gg = ln 3 / 16 gives gate = ln 3, gu = 1 / 16 gives up = 1, and y = (3/4) ln 3
    N, K = 4, 16
    w = np.full((N, K // 2), 0x22, dtype=np.uint8)
    s = np.full((N, K // 16), 0x38, dtype=np.uint8)
    x = np.full((2, K), 0x3F80, dtype=np.uint16)
    y, aux = oracle.gate_up_swiglu(w, s, LN3 / 16, w, s, 1.0 / 16, x)
    assert y.shape == (2, N)
    assert np.allclose(y, 0.75 * LN3, rtol=1e-15, atol=0)
    assert np.allclose(aux["gate"], LN3, rtol=1e-15, atol=0) and np.all(aux["up"] == 1.0)
    assert np.allclose(aux["gate_abs"], LN3, rtol=1e-15, atol=0) and np.all(aux["up_abs"] == 1.0)


@pytest.mark.parametrize("lim", [float("inf"), 0.05])
def test_gate_up_swiglu_is_the_activation_of_gate_up(lim):
    p = synth.gate_up_problem(24, 64, 3, 54)
    wg, sg, wu, su = (p[k].numpy() for k in ("wg", "sg", "wu", "su"))
    x = synth.bf16_bits(p["x"])
    y, aux = oracle.gate_up_swiglu(wg, sg, p["gg"], wu, su, p["gu"], x, lim)
    yg, ya = oracle.gemv_gate_up(wg, sg, p["gg"], wu, su, p["gu"], x)
    assert np.array_equal(aux["gate"], yg[:, :24]) and np.array_equal(aux["up"], yg[:, 24:])
    assert np.array_equal(aux["gate_abs"], ya[:, :24]) and np.array_equal(aux["up_abs"], ya[:, 24:])
    ref = np.array([[oracle.swiglu(g, u, lim) for g, u in zip(gr, ur)] for gr, ur in zip(yg[:, :24], yg[:, 24:])])
    assert np.array_equal(y, ref)
    if lim < 1:  # the limit is active for part of the outputs
        assert np.any(np.abs(yg) > lim)
    rows = [23, 0, 7]
    ys, _ = oracle.gate_up_swiglu(wg, sg, p["gg"], wu, su, p["gu"], x, lim, rows=rows)
    assert np.array_equal(ys, y[:, rows])
