"""CPU oracle for the NVFP4 weight-only GEMV (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library and its Python binding
never import it, and it imports nothing from them.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, fp64). This module only
compiles that file with the host C compiler and marshals numpy arrays through
ctypes. The GEMV functions return ``(y, yabs)``. ``y`` is the fp64 result.
``yabs`` is ``|g| * sum_k |term|``, the scale that the parity tolerance uses.
``ffn_swiglu`` returns the same pair for its down projection plus the FFN's
intermediates.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvfp4oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (host C compiler, OpenMP, -O2)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    c_i64p = ctypes.POINTER(ctypes.c_int64)
    c_u8p = ctypes.POINTER(ctypes.c_uint8)
    c_u16p = ctypes.POINTER(ctypes.c_uint16)
    c_dp = ctypes.POINTER(ctypes.c_double)
    lib.nvfp4_oracle_e2m1.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_e2m1.restype = ctypes.c_double
    lib.nvfp4_oracle_e4m3.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_e4m3.restype = ctypes.c_double
    lib.nvfp4_oracle_bf16.argtypes = [ctypes.c_uint16]
    lib.nvfp4_oracle_bf16.restype = ctypes.c_double
    lib.nvfp4_oracle_threads.argtypes = []
    lib.nvfp4_oracle_threads.restype = ctypes.c_int
    lib.nvfp4_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.nvfp4_oracle_set_threads.restype = None
    lib.nvfp4_oracle_gemv.argtypes = [c_u8p, c_u8p, ctypes.c_double, c_u16p, ctypes.c_int64,
                                      ctypes.c_int64, ctypes.c_int64, c_i64p, ctypes.c_int64,
                                      c_dp, c_dp]
    lib.nvfp4_oracle_gemv.restype = ctypes.c_int
    lib.nvfp4_oracle_gemv_gate_up.argtypes = [c_u8p, c_u8p, ctypes.c_double, c_u8p, c_u8p,
                                              ctypes.c_double, c_u16p, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int64, c_i64p,
                                              ctypes.c_int64, c_dp, c_dp]
    lib.nvfp4_oracle_gemv_gate_up.restype = ctypes.c_int
    lib.nvfp4_oracle_swiglu.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
    lib.nvfp4_oracle_swiglu.restype = ctypes.c_double
    lib.nvfp4_oracle_gate_up_swiglu.argtypes = [c_u8p, c_u8p, ctypes.c_double, c_u8p, c_u8p,
                                                ctypes.c_double, c_u16p, ctypes.c_double,
                                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                c_i64p, ctypes.c_int64, c_dp, c_dp, c_dp, c_dp, c_dp]
    lib.nvfp4_oracle_gate_up_swiglu.restype = ctypes.c_int
    lib.nvfp4_oracle_moe_gemv.argtypes = [c_u8p, c_u8p, ctypes.POINTER(ctypes.c_float),
                                          ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.c_int64, ctypes.c_int64, c_u16p, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_int64, c_i64p, ctypes.c_int64,
                                          c_dp, c_dp, c_i64p]
    lib.nvfp4_oracle_moe_gemv.restype = ctypes.c_int
    lib.nvfp4_oracle_sdict_index.argtypes = [c_u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    lib.nvfp4_oracle_sdict_index.restype = ctypes.c_int
    lib.nvfp4_oracle_sdict_idx_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    lib.nvfp4_oracle_sdict_idx_bytes.restype = ctypes.c_int64
    lib.nvfp4_oracle_gemv_sdict.argtypes = [c_u8p, c_u8p, c_u8p, ctypes.c_double, c_u16p, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, c_i64p, ctypes.c_int64, c_dp, c_dp]
    lib.nvfp4_oracle_gemv_sdict.restype = ctypes.c_int
    lib.nvfp4_oracle_moe_gemv_sdict.argtypes = [c_u8p, c_u8p, c_u8p, ctypes.POINTER(ctypes.c_float),
                                                ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                                ctypes.c_int64, ctypes.c_int64, c_u16p, ctypes.c_int,
                                                ctypes.c_int64, ctypes.c_int64, c_i64p, ctypes.c_int64,
                                                c_dp, c_dp, c_i64p]
    lib.nvfp4_oracle_moe_gemv_sdict.restype = ctypes.c_int
    lib.nvfp4_oracle_bf16_rne.argtypes = [ctypes.c_double]
    lib.nvfp4_oracle_bf16_rne.restype = ctypes.c_uint16
    lib.nvfp4_oracle_ffn_swiglu.argtypes = [c_u8p, c_u8p, ctypes.c_double, c_u8p, c_u8p, ctypes.c_double, c_u8p,
                                            c_u8p, ctypes.c_double, c_u16p, ctypes.c_double, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, c_i64p, ctypes.c_int64, c_dp, c_dp,
                                            c_dp, c_u16p, c_dp]
    lib.nvfp4_oracle_ffn_swiglu.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library. ``path`` loads another build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.uint8)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def _rows(rows):
    if rows is None:
        return None, None
    r = np.ascontiguousarray(np.asarray(rows), dtype=np.int64)
    return r, _ptr(r, ctypes.c_int64)


def e2m1(code: int, lib=None) -> float:
    return (lib or load()).nvfp4_oracle_e2m1(int(code))


def e4m3(code: int, lib=None) -> float:
    return (lib or load()).nvfp4_oracle_e4m3(int(code))


def bf16(bits: int, lib=None) -> float:
    return (lib or load()).nvfp4_oracle_bf16(int(bits) & 0xFFFF)


def threads(lib=None) -> int:
    return (lib or load()).nvfp4_oracle_threads()


def set_threads(n: int, lib=None) -> None:
    (lib or load()).nvfp4_oracle_set_threads(int(n))


def gemv(w, s, g, x_bits, rows=None, lib=None):
    """Dense oracle. w [N, K/2] u8, s [N, K/16] u8, x_bits [M, K] bf16 bit patterns.

    Returns y, yabs of shape [M, len(rows)] (all N when rows is None).
    """
    lib = lib or load()
    w, s, x = _u8(w), _u8(s), _u16(x_bits)
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    assert s.shape == (N, K // 16) and x.shape == (M, K)
    r, rp = _rows(rows)
    nr = N if r is None else r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    ya = np.empty((M, nr), dtype=np.float64)
    rc = lib.nvfp4_oracle_gemv(_ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_uint8), float(g),
                               _ptr(x, ctypes.c_uint16), M, N, K, rp, nr,
                               _ptr(y, ctypes.c_double), _ptr(ya, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemv: bad arguments")
    return y, ya


def gemv_gate_up(wg, sg, gg, wu, su, gu, x_bits, rows=None, lib=None):
    """Gate and up GEMVs of the same x; y[:, :N] = gate, y[:, N:] = up."""
    lib = lib or load()
    wg, sg, wu, su, x = _u8(wg), _u8(sg), _u8(wu), _u8(su), _u16(x_bits)
    N, K = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    assert wu.shape == wg.shape and sg.shape == su.shape == (N, K // 16)
    r, rp = _rows(rows)
    nr = 2 * N if r is None else r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    ya = np.empty((M, nr), dtype=np.float64)
    rc = lib.nvfp4_oracle_gemv_gate_up(_ptr(wg, ctypes.c_uint8), _ptr(sg, ctypes.c_uint8),
                                       float(gg), _ptr(wu, ctypes.c_uint8),
                                       _ptr(su, ctypes.c_uint8), float(gu),
                                       _ptr(x, ctypes.c_uint16), M, N, K, rp, nr,
                                       _ptr(y, ctypes.c_double), _ptr(ya, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gate_up: bad arguments")
    return y, ya


def swiglu(gate: float, up: float, lim: float = float("inf"), lib=None) -> float:
    """silu(c(gate)) * c(up) with c the clamp to [-lim, lim], in fp64."""
    return (lib or load()).nvfp4_oracle_swiglu(float(gate), float(up), float(lim))


def gate_up_swiglu(wg, sg, gg, wu, su, gu, x_bits, lim=float("inf"), rows=None, lib=None):
    """Gate/up GEMVs then the fused activation. Returns y [M, len(rows)] and a dict with the
    fp64 gate and up values and their |g| * sum |term| scales ("gate", "gate_abs", "up",
    "up_abs"), each [M, len(rows)]."""
    lib = lib or load()
    wg, sg, wu, su, x = _u8(wg), _u8(sg), _u8(wu), _u8(su), _u16(x_bits)
    N, K = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    assert wu.shape == wg.shape and sg.shape == su.shape == (N, K // 16) and x.shape == (M, K)
    r, rp = _rows(rows)
    nr = N if r is None else r.shape[0]
    out = {k: np.empty((M, nr), dtype=np.float64) for k in ("y", "gate", "gate_abs", "up", "up_abs")}
    rc = lib.nvfp4_oracle_gate_up_swiglu(_ptr(wg, ctypes.c_uint8), _ptr(sg, ctypes.c_uint8), float(gg),
                                         _ptr(wu, ctypes.c_uint8), _ptr(su, ctypes.c_uint8), float(gu),
                                         _ptr(x, ctypes.c_uint16), float(lim), M, N, K, rp, nr,
                                         *[_ptr(out[k], ctypes.c_double)
                                           for k in ("y", "gate", "gate_abs", "up", "up_abs")])
    if rc != 0:
        raise ValueError("oracle gate_up_swiglu: bad arguments")
    y = out.pop("y")
    return y, out


def moe_gemv(w, s, gs, ids, x_bits, x_per_slot, top_k, rows=None, lib=None):
    """Routed-expert oracle. w [E, N, K/2], s [E, N, K/16], gs [E] f32, ids [T*top_k] i32.

    Returns y, yabs of shape [T*top_k, len(rows)] and the count of out-of-range ids.
    """
    lib = lib or load()
    w, s, x = _u8(w), _u8(s), _u16(x_bits)
    gs = np.ascontiguousarray(np.asarray(gs), dtype=np.float32)
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), dtype=np.int32)
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 2
    assert s.shape == (E, N, K // 16) and gs.shape == (E,)
    slots = ids.shape[0]
    assert slots % top_k == 0
    T = slots // top_k
    assert x.shape == ((slots if x_per_slot else T), K)
    r, rp = _rows(rows)
    nr = N if r is None else r.shape[0]
    y = np.empty((slots, nr), dtype=np.float64)
    ya = np.empty((slots, nr), dtype=np.float64)
    bad = np.zeros(1, dtype=np.int64)
    rc = lib.nvfp4_oracle_moe_gemv(_ptr(w, ctypes.c_uint8), _ptr(s, ctypes.c_uint8),
                                   _ptr(gs, ctypes.c_float), E, _ptr(ids, ctypes.c_int32),
                                   T, top_k, _ptr(x, ctypes.c_uint16), int(bool(x_per_slot)),
                                   N, K, rp, nr, _ptr(y, ctypes.c_double),
                                   _ptr(ya, ctypes.c_double), _ptr(bad, ctypes.c_int64))
    if rc != 0:
        raise ValueError("oracle moe: bad arguments")
    return y, ya, int(bad[0])


def sdict_idx_bytes(N: int, K: int, lib=None) -> int:
    """Bytes of the index plane of one [N, K] dictionary-scaled tensor."""
    return int((lib or load()).nvfp4_oracle_sdict_idx_bytes(int(N), int(K)))


def sdict_index(idx, K: int, n: int, b: int, lib=None) -> int:
    """The 5-bit dictionary index of block b of row n (index layout in nvfp4_oracle.c)."""
    idx = _u8(idx).reshape(-1)
    return int((lib or load()).nvfp4_oracle_sdict_index(_ptr(idx, ctypes.c_uint8), int(K), int(n), int(b)))


def gemv_sdict(w, idx, sdict, g, x_bits, rows=None, lib=None):
    """Dense oracle with dictionary scales: w [N, K/2] u8, idx the packed 5-bit index plane
    (sdict_idx_bytes(N, K) bytes), sdict [32] E4M3 codes. Returns y, yabs like gemv."""
    lib = lib or load()
    w, x = _u8(w), _u16(x_bits)
    idx, sdict = _u8(idx).reshape(-1), _u8(sdict).reshape(-1)
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    assert idx.size == sdict_idx_bytes(N, K, lib) and sdict.size == 32 and x.shape == (M, K)
    r, rp = _rows(rows)
    nr = N if r is None else r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    ya = np.empty((M, nr), dtype=np.float64)
    rc = lib.nvfp4_oracle_gemv_sdict(_ptr(w, ctypes.c_uint8), _ptr(idx, ctypes.c_uint8), _ptr(sdict, ctypes.c_uint8),
                                     float(g), _ptr(x, ctypes.c_uint16), M, N, K, rp, nr,
                                     _ptr(y, ctypes.c_double), _ptr(ya, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle gemv_sdict: bad arguments")
    return y, ya


def moe_gemv_sdict(w, idx, sdict, gs, ids, x_bits, x_per_slot, top_k, rows=None, lib=None):
    """Routed-expert oracle with dictionary scales: w [E, N, K/2], idx [E, sdict_idx_bytes(N, K)],
    sdict [E, 32]. Returns y, yabs and the count of out-of-range ids, like moe_gemv."""
    lib = lib or load()
    w, x = _u8(w), _u16(x_bits)
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 2
    idx, sdict = _u8(idx).reshape(-1), _u8(sdict).reshape(-1)
    gs = np.ascontiguousarray(np.asarray(gs), dtype=np.float32)
    ids = np.ascontiguousarray(np.asarray(ids).reshape(-1), dtype=np.int32)
    assert idx.size == E * sdict_idx_bytes(N, K, lib) and sdict.size == 32 * E and gs.shape == (E,)
    slots = ids.shape[0]
    assert slots % top_k == 0
    T = slots // top_k
    assert x.shape == ((slots if x_per_slot else T), K)
    r, rp = _rows(rows)
    nr = N if r is None else r.shape[0]
    y = np.empty((slots, nr), dtype=np.float64)
    ya = np.empty((slots, nr), dtype=np.float64)
    bad = np.zeros(1, dtype=np.int64)
    rc = lib.nvfp4_oracle_moe_gemv_sdict(_ptr(w, ctypes.c_uint8), _ptr(idx, ctypes.c_uint8),
                                         _ptr(sdict, ctypes.c_uint8), _ptr(gs, ctypes.c_float), E,
                                         _ptr(ids, ctypes.c_int32), T, top_k, _ptr(x, ctypes.c_uint16),
                                         int(bool(x_per_slot)), N, K, rp, nr, _ptr(y, ctypes.c_double),
                                         _ptr(ya, ctypes.c_double), _ptr(bad, ctypes.c_int64))
    if rc != 0:
        raise ValueError("oracle moe_gemv_sdict: bad arguments")
    return y, ya, int(bad[0])


def bf16_rne(v, lib=None) -> np.ndarray:
    """fp64 values rounded to the nearest bf16, ties to even: uint16 bit patterns, same shape."""
    lib = lib or load()
    a = np.asarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    flat, o = a.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        o[i] = lib.nvfp4_oracle_bf16_rne(float(flat[i]))
    return out


def ffn_swiglu(wg, sg, gg, wu, su, gu, wd, sd, gd, x_bits, lim=float("inf"), rows=None, lib=None):
    """The FFN block: h = bf16(silu(clamp(gate)) * clamp(up)), then y = gd * W_down . h.

    wg, wu [I, H/2], sg, su [I, H/16]; wd [H, I/2], sd [H, I/16]; x_bits [M, H]. Returns y and
    yabs [M, len(rows)] (yabs: the down GEMV's |gd| * sum |term| on the bf16 h) and a dict with
    h (fp64, before rounding), h_bits (the bf16 h the down GEMV reads) and gate, gate_abs, up,
    up_abs, each [M, I]."""
    lib = lib or load()
    wg, sg, wu, su, wd, sd, x = _u8(wg), _u8(sg), _u8(wu), _u8(su), _u8(wd), _u8(sd), _u16(x_bits)
    I, H = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    assert wu.shape == wg.shape and sg.shape == su.shape == (I, H // 16) and x.shape == (M, H)
    assert wd.shape == (H, I // 2) and sd.shape == (H, I // 16)
    r, rp = _rows(rows)
    nr = H if r is None else r.shape[0]
    y = np.empty((M, nr), dtype=np.float64)
    ya = np.empty((M, nr), dtype=np.float64)
    h = np.empty((M, I), dtype=np.float64)
    hb = np.empty((M, I), dtype=np.uint16)
    aux = np.empty((4, M, I), dtype=np.float64)
    rc = lib.nvfp4_oracle_ffn_swiglu(_ptr(wg, ctypes.c_uint8), _ptr(sg, ctypes.c_uint8), float(gg),
                                     _ptr(wu, ctypes.c_uint8), _ptr(su, ctypes.c_uint8), float(gu),
                                     _ptr(wd, ctypes.c_uint8), _ptr(sd, ctypes.c_uint8), float(gd),
                                     _ptr(x, ctypes.c_uint16), float(lim), M, H, I, rp, nr,
                                     _ptr(y, ctypes.c_double), _ptr(ya, ctypes.c_double),
                                     _ptr(h, ctypes.c_double), _ptr(hb, ctypes.c_uint16),
                                     _ptr(aux, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle ffn_swiglu: bad arguments")
    out = {"h": h, "h_bits": hb, "gate": aux[0], "gate_abs": aux[1], "up": aux[2], "up_abs": aux[3]}
    return y, ya, out
