"""The oracle's pins catch plausible mistakes.

Each case copies the oracle's C source and plants one mistake in the copy: a
swapped nibble order, a dropped sign, a wrong exponent bias, a wrong scale
index, a dropped term, a transposed operand, and so on. It then builds the copy
into a scratch library and checks that the pin battery below rejects it. The
unmodified source must pass the same battery. Everything runs on the CPU.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from nvfp4_weight_only_gemv_gb300 import synth

from test_oracle_pins import E2M1_TABLE, _arrays, _golden, dequant, torch_bf16, torch_e4m3
from test_oracle_sdict import _golden as _sdict_golden, pack_indices, random_case
from test_oracle_ffn import hand_worked_ffn

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.c")

MUTANTS = {
    "nibble_order": ("(wrow[k / 2] >> (4 * (k & 1)))", "(wrow[k / 2] >> (4 * (1 - (k & 1))))", 1),
    "e2m1_sign_dropped": ("return sign ? -mag : mag;", "return mag;", 1),
    "e2m1_bias": ("exp_field - 1)", "exp_field - 2)", 1),
    "e2m1_subnormal": ("mag = 0.5 * (double)mant;", "mag = 1.0 * (double)mant;", 1),
    "e4m3_bias": ("exp_field - 7)", "exp_field - 8)", 1),
    "e4m3_subnormal": ("ldexp((double)mant / 8.0, -6)", "ldexp((double)mant / 8.0, -7)", 1),
    "e4m3_no_nan": ("if (exp_field == 15 && mant == 7) return NAN;", "", 1),
    "scale_index": ("srow[k / 16]", "srow[k / 32]", 1),
    "scale_row_stride": ("const uint8_t *srow = s + n * (K / 16);", "const uint8_t *srow = s + n * (K / 32);", 1),
    "global_scale_dropped": ("y[m * nrows + i] = g * sum;", "y[m * nrows + i] = sum;", 1),
    "x_row_transposed": ("dot_row(wrow, srow, x + m * K, K, &sum, &abs_sum);",
                         "dot_row(wrow, srow, x + m, K, &sum, &abs_sum);", 1),
    "dropped_last_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k < K - 1; ++k)", 1),
    "gate_up_swapped": ("int up = r >= N;", "int up = r < N;", 1),
    "moe_x_row": ("int64_t xrow = x_per_slot ? sl : sl / top_k;", "int64_t xrow = x_per_slot ? sl : 0;", 1),
    "moe_global_scale": ("double g = (double)gs[e];", "double g = (double)gs[0];", 1),
    "silu_sign": ("gc / (1.0 + exp(-gc))", "gc / (1.0 + exp(gc))", 1),
    "silu_one_dropped": ("gc / (1.0 + exp(-gc))", "gc / exp(-gc)", 1),
    "gate_clamp_dropped": ("double gc = gate > lim ? lim : (gate < -lim ? -lim : gate);", "double gc = gate;", 1),
    "up_clamp_one_sided": ("double uc = up > lim ? lim : (up < -lim ? -lim : up);",
                           "double uc = up > lim ? lim : up;", 1),
    "swiglu_args_swapped": ("y[m * nrows + i] = nvfp4_oracle_swiglu(gv, uv, lim);",
                            "y[m * nrows + i] = nvfp4_oracle_swiglu(uv, gv, lim);", 1),
    "swiglu_up_scale": ("double gv = gg * sg_sum, uv = gu * su_sum;", "double gv = gg * sg_sum, uv = gg * su_sum;", 1),
    "sdict_index_width": ("    for (int i = 0; i < 5; ++i) {\n        int64_t bit", "    for (int i = 0; i < 4; ++i) {\n        int64_t bit", 1),
    "sdict_index_stride": ("int64_t bit = 5 * q + i;", "int64_t bit = 6 * q + i;", 1),
    "sdict_bit_order": ("v |= ((rec[bit / 8] >> (bit % 8)) & 1) << i;", "v |= ((rec[bit / 8] >> (7 - bit % 8)) & 1) << i;", 1),
    "sdict_table_offset": ("srow[b] = dict[nvfp4_oracle_sdict_index(idx, K, n, b)];",
                           "srow[b] = dict[(nvfp4_oracle_sdict_index(idx, K, n, b) + 1) & 31];", 1),
    "sdict_position_transposed": ("int64_t q = (n % 16) * 16 + (b % 16);", "int64_t q = (b % 16) * 16 + (n % 16);", 1),
    "sdict_record_order": ("((n / 16) * (K / 256) + b / 16) * 160", "((b / 16) * (K / 256) + n / 16) * 160", 1),
    "sdict_moe_plane": ("sdict_scale_row(idx + e * plane, dict + 32 * e, K, n, sr);",
                        "sdict_scale_row(idx, dict + 32 * e, K, n, sr);", 1),
    "sdict_moe_table": ("sdict_scale_row(idx + e * plane, dict + 32 * e, K, n, sr);",
                        "sdict_scale_row(idx + e * plane, dict, K, n, sr);", 1),
    "bf16_ties_away": ("double m = rint(a / q);", "double m = round(a / q);", 1),
    "bf16_truncates": ("double m = rint(a / q);", "double m = floor(a / q);", 1),
    "bf16_mantissa_bits": ("ldexp(1.0, ex - 7)", "ldexp(1.0, ex - 8)", 1),
    "bf16_subnormal_step": ("ldexp(1.0, -133)", "ldexp(1.0, -134)", 1),
    "bf16_sign_dropped": ("return sign | (uint16_t)(u >> 16);", "return (uint16_t)(u >> 16);", 1),
    "ffn_h_truncated": ("hb[j] = nvfp4_oracle_bf16_rne(h[j]);",
                        "{ float f = (float)h[j]; uint32_t u; memcpy(&u, &f, 4); hb[j] = (uint16_t)(u >> 16); }", 1),
    "ffn_down_scale": ("rc = nvfp4_oracle_gemv(wd, sd, gd, hb,", "rc = nvfp4_oracle_gemv(wd, sd, gg, hb,", 1),
    "ffn_gate_up_swapped": ("nvfp4_oracle_gate_up_swiglu(wg, sg, gg, wu, su, gu, x, lim, M, I, H,",
                            "nvfp4_oracle_gate_up_swiglu(wu, su, gu, wg, sg, gg, x, lim, M, I, H,", 1),
}


def battery(lib):
    """Return the names of the pins that ``lib`` fails (empty when all hold)."""
    fails = []
    if any(oracle.e2m1(c, lib) != E2M1_TABLE[c] or
           np.signbit(oracle.e2m1(c, lib)) != np.signbit(E2M1_TABLE[c]) for c in range(16)):
        fails.append("e2m1")
    ref = torch_e4m3(np.arange(256))
    got = np.array([oracle.e4m3(c, lib) for c in range(256)])
    if not np.array_equal(np.isnan(got), np.isnan(ref)) or \
            not np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)]):
        fails.append("e4m3")
    for ex in _golden("hand_worked.json")["examples"]:
        w, s, x = _arrays(ex)
        y, _ = oracle.gemv(w, s, ex["g"], x, lib=lib)
        if not np.array_equal(y, np.array(ex["y"])):
            fails.append("hand_worked:" + ex["name"])
    p = synth.dense_problem(48, 160, 3, 51)
    w, s, x = p["w"].numpy(), p["s"].numpy(), synth.bf16_bits(p["x"])
    y, ya = oracle.gemv(w, s, p["g"], x, lib=lib)
    refd = p["g"] * (torch_bf16(x) @ dequant(w, s).T)
    if not np.all(np.abs(y - refd) <= 1e-12 * np.maximum(ya, 1e-300)):
        fails.append("numpy_matmul")
    q = synth.gate_up_problem(24, 64, 2, 52)
    wg, sg, wu, su = (q[k].numpy() for k in ("wg", "sg", "wu", "su"))
    xq = synth.bf16_bits(q["x"])
    y, ya = oracle.gemv_gate_up(wg, sg, q["gg"], wu, su, q["gu"], xq, lib=lib)
    xv = torch_bf16(xq)
    refg = np.concatenate([q["gg"] * (xv @ dequant(wg, sg).T), q["gu"] * (xv @ dequant(wu, su).T)], 1)
    if not np.all(np.abs(y - refg) <= 1e-12 * np.maximum(ya, 1e-300)):
        fails.append("gate_up")
    for xps in (False, True):
        r = synth.moe_problem(9, 16, 48, 3, 3, xps, seed=53)
        wm, sm, gs, ids = r["w"].numpy(), r["s"].numpy(), r["gs"].numpy(), r["ids"].numpy()
        xm = synth.bf16_bits(r["x"])
        y, ya, _ = oracle.moe_gemv(wm, sm, gs, ids, xm, xps, 3, lib=lib)
        xv = torch_bf16(xm)
        for sl in range(9):
            e = ids[sl]
            refm = float(gs[e]) * (dequant(wm[e], sm[e]) @ xv[sl if xps else sl // 3])
            if not np.all(np.abs(y[sl] - refm) <= 1e-12 * np.maximum(ya[sl], 1e-300)):
                fails.append(f"moe(x_per_slot={xps})")
                break
    # the fused activation: closed forms of the logistic function, the clamp, and the hand-worked
    # gate/up example (gate = ln 3, up = 1); see the pins of the same names
    ln3 = math.log(3.0)
    if not (math.isclose(oracle.swiglu(ln3, 1.0, lib=lib), 0.75 * ln3, rel_tol=1e-15) and
            math.isclose(oracle.swiglu(-ln3, 1.0, lib=lib), -0.25 * ln3, rel_tol=1e-15)):
        fails.append("silu_closed_form")
    if not (oracle.swiglu(5.0, 1.0, 2.0, lib=lib) == oracle.swiglu(2.0, 1.0, lib=lib) and
            oracle.swiglu(1.0, -9.0, 2.0, lib=lib) == oracle.swiglu(1.0, -2.0, lib=lib)):
        fails.append("swiglu_clamp")
    w1 = np.full((4, 8), 0x22, dtype=np.uint8)
    s1 = np.full((4, 1), 0x38, dtype=np.uint8)
    x1 = np.full((1, 16), 0x3F80, dtype=np.uint16)
    y1, _ = oracle.gate_up_swiglu(w1, s1, ln3 / 16, w1, s1, 1.0 / 16, x1, lib=lib)
    y2, _ = oracle.gate_up_swiglu(w1, s1, 1.0 / 16, w1, s1, ln3 / 16, x1, lib=lib)
    if not (np.allclose(y1, 0.75 * ln3, rtol=1e-15, atol=0) and
            np.allclose(y2, ln3 / (1.0 + math.exp(-1.0)), rtol=1e-15, atol=0)):
        fails.append("gate_up_swiglu_hand_worked")
    # the dictionary form: hand-worked layouts, and exact equality with the plain form (dense,
    # ragged N; routed experts with a table and index plane per expert)
    for ex in _sdict_golden()["examples"]:
        N, K = ex["N"], ex["K"]
        wd = np.frombuffer(bytes.fromhex(ex["w_row"]) * N, dtype=np.uint8).reshape(N, K // 2)
        idx = np.frombuffer(bytes.fromhex(ex["idx"]), dtype=np.uint8)
        sd = np.array([int(v, 16) for v in ex["dict"]], dtype=np.uint8)
        xd = np.full((ex["M"], K), int(ex["x_value"], 16), dtype=np.uint16)
        y, _ = oracle.gemv_sdict(wd, idx, sd, ex["g"], xd, lib=lib)
        if not np.array_equal(y, np.array([ex["y"]])):
            fails.append("sdict_hand_worked:" + ex["name"])
    wd, sd, ind, xd = random_case(40, 512, 2, 61)
    y, _ = oracle.gemv_sdict(wd, pack_indices(ind, 40, 512), sd, 0.5, xd, lib=lib)
    yp, _ = oracle.gemv(wd, sd[ind].astype(np.uint8), 0.5, xd, lib=lib)
    if not np.array_equal(y, yp):
        fails.append("sdict_equals_plain")
    rng = np.random.default_rng(62)
    E, N, K = 3, 20, 256
    wm = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    sdm = np.stack([rng.permutation(np.arange(0x20, 0x60))[:32] for _ in range(E)]).astype(np.uint8)
    indm = rng.integers(0, 32, (E, N, K // 16))
    planes = np.stack([pack_indices(indm[e], N, K) for e in range(E)])
    sm = np.stack([sdm[e][indm[e]] for e in range(E)]).astype(np.uint8)
    gs = np.array([0.5, 1.0, 2.0], dtype=np.float32)
    ids = np.array([2, 0, 1, 2], dtype=np.int32)
    xm = synth.bf16_bits(synth.random_x(2, K, 63))
    y, _, _ = oracle.moe_gemv_sdict(wm, planes, sdm, gs, ids, xm, False, 2, lib=lib)
    yp, _, _ = oracle.moe_gemv(wm, sm, gs, ids, xm, False, 2, lib=lib)
    if not np.array_equal(y, yp):
        fails.append("sdict_moe_equals_plain")
    # bf16 rounding of the FFN's h: round trips, ties to even, PyTorch's float32 conversion, and
    # the FFN's closed form (see test_oracle_ffn.py)
    bits = np.arange(0, 0x7F80, 61, dtype=np.uint16)
    vals = np.array([oracle.bf16(int(b), lib) for b in bits])
    if not np.array_equal(oracle.bf16_rne(-vals, lib), bits | 0x8000):
        fails.append("bf16_round_trip")
    lo = np.arange(0, 0x7F7F, 37, dtype=np.int64)
    mid = (np.array([oracle.bf16(int(b), lib) for b in lo]) + np.array([oracle.bf16(int(b) + 1, lib) for b in lo])) / 2
    if not np.array_equal(oracle.bf16_rne(mid, lib).astype(np.int64), np.where(lo % 2 == 0, lo, lo + 1)):
        fails.append("bf16_ties_to_even")
    v = np.random.default_rng(64).standard_normal(4000).astype(np.float32) * np.float32(3.0)
    v = np.concatenate([v, np.float32(2.0 ** -140) * v[:500]])
    if not np.array_equal(oracle.bf16_rne(v.astype(np.float64), lib),
                          torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)):
        fails.append("bf16_vs_pytorch")
    y, y_exp, hb, hb_exp, _, _ = hand_worked_ffn(lib)
    if not (np.array_equal(y, y_exp) and np.array_equal(hb, hb_exp)):
        fails.append("ffn_hand_worked")
    return fails


def test_unmodified_oracle_passes_battery():
    assert battery(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new, count = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= count, f"mutation site for {name} not found"
    mutated = src.replace(old, new, count)
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(mutated)
    so = str(tmp_path / f"libmutant_{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", so, str(path),
                    "-lm"], check=True, capture_output=True)
    fails = battery(oracle.load(so))
    assert fails, f"mutant {name} passed every pin"
