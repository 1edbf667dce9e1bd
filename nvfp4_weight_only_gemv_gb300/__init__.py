"""NVFP4 (nvfp4/g16) weight-only GEMV for GB300: thin Python binding over ``libnvfp4gemv.so``.

Every function here only checks tensors and passes pointers, sizes and the current CUDA
stream to the C ABI declared in ``include/nvfp4_gemv.h``. All arithmetic runs in that
library's CUDA kernels. There is no CPU or PyTorch fallback. If the library cannot be
loaded, every call raises.

Tensors (CUDA, contiguous):
  w  uint8 [N, K/2]   E2M1 codes, element 2j in the low nibble of byte j
  s  uint8 [N, K/16]  E4M3 block scales
  x  bfloat16 [M, K]  activations, M <= 8
  y  float32 or bfloat16 [M, N]
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = ["gemv", "gemv_gate_up", "gemv_gate_up_swiglu", "ffn_swiglu", "ffn_swiglu_static", "ffn_workspace",
           "ffn_workspace_bytes",
           "moe_gemv", "gemv_sdict", "moe_gemv_sdict",
           "sdict_plane_bytes", "sdict_encode", "device_status", "set_wait_budget_ns",
           "set_variant", "set_pdl", "fp32_fallbacks", "phase_trace", "describe_plan", "describe_plan_host", "library", "library_path", "NVFP4Error",
           "OUT_F32", "OUT_BF16", "DEV_TIMEOUT", "DEV_BAD_EXPERT", "DEV_INTERNAL"]

OUT_F32 = 0
OUT_BF16 = 1
DEV_TIMEOUT = 1
DEV_BAD_EXPERT = 2
DEV_INTERNAL = 4

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    """The library this process loads: NVFP4_GEMV_LIBRARY if set (a diagnostic or experiment
    build of the same source), else the in-tree build."""
    return os.environ.get("NVFP4_GEMV_LIBRARY") or _build.LIB_PATH


def _declare(lib):
    vp, u8p, u16p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    i32 = ctypes.c_int
    lib.nvfp4_gemv.argtypes = [u8p, u8p, ctypes.c_float, u16p, vp, i32, i32, i32, i32, vp]
    lib.nvfp4_gemv.restype = i32
    lib.nvfp4_gemv_gate_up.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u16p, vp,
                                       i32, i32, i32, i32, vp]
    lib.nvfp4_gemv_gate_up.restype = i32
    lib.nvfp4_gemv_gate_up_swiglu.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u16p,
                                              ctypes.c_float, vp, i32, i32, i32, i32, vp]
    lib.nvfp4_ffn_swiglu.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float,
                                     u16p, ctypes.c_float, vp, vp, i32, i32, i32, i32, vp]
    lib.nvfp4_ffn_swiglu.restype = i32
    lib.nvfp4_ffn_swiglu_static.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u8p, u8p,
                                            ctypes.c_float, u16p, ctypes.c_float, vp, i32, i32, i32, i32, vp]
    lib.nvfp4_ffn_swiglu_static.restype = i32
    lib.nvfp4_ffn_workspace_bytes.argtypes = [i32, i32]
    lib.nvfp4_ffn_workspace_bytes.restype = ctypes.c_int64
    lib.nvfp4_gemv_gate_up_swiglu.restype = i32
    lib.nvfp4_moe_gemv.argtypes = [u8p, u8p, vp, i32, vp, i32, i32, u16p, i32, vp, i32, i32, i32,
                                   vp, vp]
    lib.nvfp4_moe_gemv.restype = i32
    lib.nvfp4_status_string.argtypes = [i32]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_last_cuda_error.argtypes = []
    lib.nvfp4_last_cuda_error.restype = i32
    lib.nvfp4_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
    lib.nvfp4_device_status.restype = i32
    lib.nvfp4_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
    lib.nvfp4_set_wait_budget_ns.restype = None
    lib.nvfp4_set_variant.argtypes = [i32]
    lib.nvfp4_set_variant.restype = None
    lib.nvfp4_set_pdl.argtypes = [i32]
    lib.nvfp4_set_pdl.restype = None
    lib.nvfp4_fp32_fallbacks.argtypes = [vp]
    lib.nvfp4_fp32_fallbacks.restype = ctypes.c_longlong
    lib.nvfp4_describe_plan.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.c_char_p, i32]
    lib.nvfp4_describe_plan.restype = i32
    lib.nvfp4_describe_plan_host.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, ctypes.c_char_p, i32]
    lib.nvfp4_describe_plan_host.restype = i32
    lib.nvfp4_gemv_sdict.argtypes = [u8p, u8p, u8p, ctypes.c_float, u16p, vp, i32, i32, i32, i32, vp]
    lib.nvfp4_gemv_sdict.restype = i32
    lib.nvfp4_moe_gemv_sdict.argtypes = [u8p, u8p, u8p, vp, i32, vp, i32, i32, u16p, i32, vp, i32, i32, i32, vp, vp]
    lib.nvfp4_moe_gemv_sdict.restype = i32
    lib.nvfp4_sdict_plane_bytes.argtypes = [i32, i32]
    lib.nvfp4_sdict_plane_bytes.restype = ctypes.c_int64
    lib.nvfp4_sdict_encode.argtypes = [vp, i32, i32, vp, vp]
    lib.nvfp4_sdict_encode.restype = i32
    lib.nvfp4_phase_trace.argtypes = [vp, i32, vp]
    lib.nvfp4_phase_trace.restype = i32
    lib.nvfp4_version.argtypes = []
    lib.nvfp4_version.restype = i32
    return lib


def library(build_if_missing: bool = True):
    """The loaded ctypes library (built first when missing or stale and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if build_if_missing and path == _build.LIB_PATH and _build.is_stale():
                try:
                    _build.build()
                except RuntimeError:
                    if not os.path.exists(path):
                        raise
            if not os.path.exists(path):
                raise RuntimeError(f"NVFP4 GEMV CUDA library not found at {path}; run "
                                   "`python -m nvfp4_weight_only_gemv_gb300.build`")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def status_string(status: int) -> str:
    try:
        return library(build_if_missing=False).nvfp4_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return "unknown"


def _check(status: int, what: str):
    if status != 0:
        raise NVFP4Error(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _one_device(*tensors):
    """The kernels run on the current CUDA device and read every operand there."""
    dev = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.device.index != dev:
            raise ValueError(f"every tensor must be on the current CUDA device cuda:{dev} (got {t.device})")


def _out(out, shape, out_dtype, device):
    """The output tensor: ``out`` when given (its own dtype wins), else a new one."""
    if out is None:
        return torch.empty(shape, dtype=out_dtype, device=device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"out must be float32 or bfloat16 (got {out.dtype})")
    _need(out, "out", out.dtype, len(shape))
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must have shape {tuple(shape)} (got {tuple(out.shape)})")
    return out


def _out_code(dtype) -> int:
    if dtype == torch.float32:
        return OUT_F32
    if dtype == torch.bfloat16:
        return OUT_BF16
    raise TypeError("out_dtype must be torch.float32 or torch.bfloat16")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(t.data_ptr() or 16)


def gemv(w: torch.Tensor, s: torch.Tensor, g: float, x: torch.Tensor, out=None,
         out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """y[M, N] = g * dequant(w, s) @ x^T on the current (or given) CUDA stream."""
    _need(w, "w", torch.uint8, 2)
    _need(s, "s", torch.uint8, 2)
    _need(x, "x", torch.bfloat16, 2)
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    if tuple(s.shape) != (N, K // 16) or x.shape[1] != K:
        raise ValueError(f"shape mismatch: w {tuple(w.shape)}, s {tuple(s.shape)}, x {tuple(x.shape)}")
    y = _out(out, (M, N), out_dtype, x.device)
    _one_device(w, s, x, y)
    st = library().nvfp4_gemv(_ptr(w), _ptr(s), float(g), _ptr(x), _ptr(y), _out_code(y.dtype),
                              M, N, K, ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_gemv")
    return y


def gemv_gate_up(wg, sg, gg, wu, su, gu, x, out=None, out_dtype=torch.float32,
                 stream=None) -> torch.Tensor:
    """y[M, 2N] = [gg * W_gate . x | gu * W_up . x] in one launch."""
    for t, n in ((wg, "w_gate"), (wu, "w_up")):
        _need(t, n, torch.uint8, 2)
    for t, n in ((sg, "s_gate"), (su, "s_up")):
        _need(t, n, torch.uint8, 2)
    _need(x, "x", torch.bfloat16, 2)
    N, K = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    if tuple(wu.shape) != tuple(wg.shape) or tuple(sg.shape) != (N, K // 16) or \
            tuple(su.shape) != (N, K // 16) or x.shape[1] != K:
        raise ValueError("shape mismatch between gate, up and x")
    y = _out(out, (M, 2 * N), out_dtype, x.device)
    _one_device(wg, sg, wu, su, x, y)
    st = library().nvfp4_gemv_gate_up(_ptr(wg), _ptr(sg), float(gg), _ptr(wu), _ptr(su), float(gu),
                                      _ptr(x), _ptr(y), _out_code(y.dtype), M, N, K,
                                      ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_gemv_gate_up")
    return y


def gemv_gate_up_swiglu(wg, sg, gg, wu, su, gu, x, clamp_limit: float = float("inf"), out=None,
                        out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    """y[M, N] = silu(c(gg * W_gate . x)) * c(gu * W_up . x), c = clamp to [-clamp_limit,
    clamp_limit] (inf: none), in one launch; the gate|up product is never written."""
    for t, n in ((wg, "w_gate"), (wu, "w_up")):
        _need(t, n, torch.uint8, 2)
    for t, n in ((sg, "s_gate"), (su, "s_up")):
        _need(t, n, torch.uint8, 2)
    _need(x, "x", torch.bfloat16, 2)
    N, K = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    if tuple(wu.shape) != tuple(wg.shape) or tuple(sg.shape) != (N, K // 16) or \
            tuple(su.shape) != (N, K // 16) or x.shape[1] != K:
        raise ValueError("shape mismatch between gate, up and x")
    y = _out(out, (M, N), out_dtype, x.device)
    _one_device(wg, sg, wu, su, x, y)
    st = library().nvfp4_gemv_gate_up_swiglu(_ptr(wg), _ptr(sg), float(gg), _ptr(wu), _ptr(su), float(gu),
                                             _ptr(x), float(clamp_limit), _ptr(y), _out_code(y.dtype),
                                             M, N, K, ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_gemv_gate_up_swiglu")
    return y


def ffn_workspace_bytes(M: int, I: int) -> int:
    """Bytes of workspace ffn_swiglu needs for M rows and intermediate size I."""
    n = int(library().nvfp4_ffn_workspace_bytes(int(M), int(I)))
    if n < 0:
        raise ValueError(f"no FFN workspace for M={M}, I={I}")
    return n


def ffn_workspace(M: int, I: int, device=None) -> torch.Tensor:
    """A zeroed workspace for ffn_swiglu (uint8, 256-byte aligned by the caching allocator).
    Reuse it across calls: every call leaves its counters at zero for the next."""
    return torch.zeros(ffn_workspace_bytes(M, I), dtype=torch.uint8, device=device or "cuda")


def ffn_swiglu(wg, sg, gg, wu, su, gu, wd, sd, gd, x, clamp_limit: float = float("inf"), workspace=None,
               out=None, out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """The FFN block: h = bf16(silu(c(gg * W_gate . x)) * c(gu * W_up . x)), y = gd * W_down . h.

    wg, wu uint8 [I, H/2], sg, su [I, H/16]; wd [H, I/2], sd [H, I/16]; x bf16 [M, H]; y [M, H].
    ``workspace`` (from ffn_workspace) holds the launch's counters and h (bf16 [M, I] at byte
    2048); None allocates a zeroed one for this call. Calls sharing a workspace must be ordered."""
    for t, n in ((wg, "w_gate"), (wu, "w_up"), (wd, "w_down")):
        _need(t, n, torch.uint8, 2)
    for t, n in ((sg, "s_gate"), (su, "s_up"), (sd, "s_down")):
        _need(t, n, torch.uint8, 2)
    _need(x, "x", torch.bfloat16, 2)
    I, H = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    if tuple(wu.shape) != tuple(wg.shape) or tuple(sg.shape) != (I, H // 16) or \
            tuple(su.shape) != (I, H // 16) or x.shape[1] != H:
        raise ValueError("shape mismatch between gate, up and x")
    if tuple(wd.shape) != (H, I // 2) or tuple(sd.shape) != (H, I // 16):
        raise ValueError("down weight must be [H, I/2] with scales [H, I/16]")
    if workspace is None:
        workspace = ffn_workspace(M, I, x.device)
    _need(workspace, "workspace", torch.uint8, 1)
    if workspace.numel() < ffn_workspace_bytes(M, I):
        raise ValueError("workspace too small")
    y = _out(out, (M, H), out_dtype, x.device)
    _one_device(wg, sg, wu, su, wd, sd, x, workspace, y)
    st = library().nvfp4_ffn_swiglu(_ptr(wg), _ptr(sg), float(gg), _ptr(wu), _ptr(su), float(gu), _ptr(wd),
                                    _ptr(sd), float(gd), _ptr(x), float(clamp_limit), _ptr(workspace), _ptr(y),
                                    _out_code(y.dtype), M, H, I, ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_ffn_swiglu")
    return y


def ffn_swiglu_static(wg, sg, gg, wu, su, gu, wd, sd, gd, x, clamp_limit: float = float("inf"), out=None,
                      out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """ffn_swiglu with the library's own 256 KB device array as the workspace (nothing allocated
    by the caller). Calls on a device share that array: they must not overlap in time."""
    for t, n in ((wg, "w_gate"), (wu, "w_up"), (wd, "w_down")):
        _need(t, n, torch.uint8, 2)
    for t, n in ((sg, "s_gate"), (su, "s_up"), (sd, "s_down")):
        _need(t, n, torch.uint8, 2)
    _need(x, "x", torch.bfloat16, 2)
    I, H = wg.shape[0], wg.shape[1] * 2
    M = x.shape[0]
    if tuple(wu.shape) != tuple(wg.shape) or tuple(sg.shape) != (I, H // 16) or \
            tuple(su.shape) != (I, H // 16) or x.shape[1] != H:
        raise ValueError("shape mismatch between gate, up and x")
    if tuple(wd.shape) != (H, I // 2) or tuple(sd.shape) != (H, I // 16):
        raise ValueError("down weight must be [H, I/2] with scales [H, I/16]")
    y = _out(out, (M, H), out_dtype, x.device)
    _one_device(wg, sg, wu, su, wd, sd, x, y)
    st = library().nvfp4_ffn_swiglu_static(_ptr(wg), _ptr(sg), float(gg), _ptr(wu), _ptr(su), float(gu), _ptr(wd),
                                           _ptr(sd), float(gd), _ptr(x), float(clamp_limit), _ptr(y),
                                           _out_code(y.dtype), M, H, I, ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_ffn_swiglu_static")
    return y


def moe_gemv(w, s, gs, ids, x, x_per_slot: bool, top_k: int, out=None, out_dtype=torch.float32,
             status=None, stream=None) -> torch.Tensor:
    """Routed-expert GEMV: y[T*top_k, N]; slot t*top_k+j uses expert ids[t*top_k+j].

    w uint8 [E, N, K/2], s uint8 [E, N, K/16], gs float32 [E], ids int32 [T*top_k],
    x bf16 [T, K] (x_per_slot False) or [T*top_k, K] (True). ``status`` is an optional
    int32 CUDA tensor of one element that receives device status bits.
    """
    _need(w, "w", torch.uint8, 3)
    _need(s, "s", torch.uint8, 3)
    _need(gs, "global_scales", torch.float32, 1)
    _need(ids, "expert_ids", torch.int32, 1)
    _need(x, "x", torch.bfloat16, 2)
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 2
    slots = ids.shape[0]
    if top_k <= 0 or slots % top_k:
        raise ValueError("expert_ids length must be a multiple of top_k")
    T = slots // top_k
    rows = slots if x_per_slot else T
    if tuple(s.shape) != (E, N, K // 16) or gs.shape[0] != E or tuple(x.shape) != (rows, K):
        raise ValueError("shape mismatch in moe_gemv arguments")
    if status is not None:
        _need(status, "status", torch.int32, 1)
    y = _out(out, (slots, N), out_dtype, x.device)
    _one_device(w, s, gs, ids, x, y, status)
    st = library().nvfp4_moe_gemv(_ptr(w), _ptr(s), _ptr(gs), E, _ptr(ids), T, top_k, _ptr(x),
                                  int(bool(x_per_slot)), _ptr(y), _out_code(y.dtype), N, K,
                                  ctypes.c_void_p(status.data_ptr()) if status is not None else None,
                                  ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_moe_gemv")
    return y


def sdict_plane_bytes(N: int, K: int) -> int:
    """Bytes of the dictionary index plane of one [N, K] weight (K % 256 == 0)."""
    n = library(build_if_missing=False).nvfp4_sdict_plane_bytes(int(N), int(K))
    if n < 0:
        raise ValueError("dictionary scales need N >= 0 and K % 256 == 0")
    return int(n)


def sdict_encode(s: torch.Tensor):
    """Dictionary form of plain E4M3 block scales s uint8 [N, K/16] (or [E, N, K/16], one
    dictionary per expert), on the host: returns (index plane uint8 [sdict_plane_bytes(N, K)]
    ([E, ...] for experts), table uint8 [32] ([E, 32])) as CPU tensors. Raises ValueError when
    a tensor's scales take more than 32 distinct codes (it has no dictionary form)."""
    if s.dtype != torch.uint8 or s.dim() not in (2, 3):
        raise TypeError("s must be a uint8 tensor [N, K/16] or [E, N, K/16]")
    src = s.detach().to("cpu").contiguous()
    experts = src.unsqueeze(0) if src.dim() == 2 else src
    N, K = experts.shape[1], experts.shape[2] * 16
    lib = library(build_if_missing=False)
    planes = torch.zeros(experts.shape[0], sdict_plane_bytes(N, K), dtype=torch.uint8)
    tables = torch.zeros(experts.shape[0], 32, dtype=torch.uint8)
    for e in range(experts.shape[0]):
        rc = lib.nvfp4_sdict_encode(ctypes.c_void_p(experts[e].data_ptr()), N, K, ctypes.c_void_p(planes[e].data_ptr()),
                                    ctypes.c_void_p(tables[e].data_ptr()))
        if rc == -1:
            raise ValueError(f"tensor {e}: more than 32 distinct scale codes (no dictionary form)")
        if rc < 0:
            raise ValueError("sdict_encode: bad arguments")
    if src.dim() == 2:
        return planes[0], tables[0]
    return planes, tables


def gemv_sdict(w: torch.Tensor, idx: torch.Tensor, sdict: torch.Tensor, g: float, x: torch.Tensor, out=None,
               out_dtype=torch.float32, stream=None) -> torch.Tensor:
    """gemv with dictionary scales: w uint8 [N, K/2], idx uint8 index plane [sdict_plane_bytes(N, K)],
    sdict uint8 [32] E4M3 codes."""
    _need(w, "w", torch.uint8, 2)
    _need(idx, "idx", torch.uint8, 1)
    _need(sdict, "sdict", torch.uint8, 1)
    _need(x, "x", torch.bfloat16, 2)
    N, K = w.shape[0], w.shape[1] * 2
    M = x.shape[0]
    if idx.numel() != sdict_plane_bytes(N, K) or sdict.numel() != 32 or x.shape[1] != K:
        raise ValueError(f"shape mismatch: w {tuple(w.shape)}, idx {tuple(idx.shape)}, sdict {tuple(sdict.shape)}, "
                         f"x {tuple(x.shape)}")
    y = _out(out, (M, N), out_dtype, x.device)
    _one_device(w, idx, sdict, x, y)
    st = library().nvfp4_gemv_sdict(_ptr(w), _ptr(idx), _ptr(sdict), float(g), _ptr(x), _ptr(y), _out_code(y.dtype),
                                    M, N, K, ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_gemv_sdict")
    return y


def moe_gemv_sdict(w, idx, sdict, gs, ids, x, x_per_slot: bool, top_k: int, out=None, out_dtype=torch.float32,
                   status=None, stream=None) -> torch.Tensor:
    """moe_gemv with dictionary scales: idx uint8 [E, sdict_plane_bytes(N, K)], sdict uint8 [E, 32]."""
    _need(w, "w", torch.uint8, 3)
    _need(idx, "idx", torch.uint8, 2)
    _need(sdict, "sdict", torch.uint8, 2)
    _need(gs, "global_scales", torch.float32, 1)
    _need(ids, "expert_ids", torch.int32, 1)
    _need(x, "x", torch.bfloat16, 2)
    E, N, K = w.shape[0], w.shape[1], w.shape[2] * 2
    slots = ids.shape[0]
    if top_k <= 0 or slots % top_k:
        raise ValueError("expert_ids length must be a multiple of top_k")
    T = slots // top_k
    rows = slots if x_per_slot else T
    if (tuple(idx.shape) != (E, sdict_plane_bytes(N, K)) or tuple(sdict.shape) != (E, 32) or gs.shape[0] != E
            or tuple(x.shape) != (rows, K)):
        raise ValueError("shape mismatch in moe_gemv_sdict arguments")
    if status is not None:
        _need(status, "status", torch.int32, 1)
    y = _out(out, (slots, N), out_dtype, x.device)
    _one_device(w, idx, sdict, gs, ids, x, y, status)
    st = library().nvfp4_moe_gemv_sdict(_ptr(w), _ptr(idx), _ptr(sdict), _ptr(gs), E, _ptr(ids), T, top_k, _ptr(x),
                                        int(bool(x_per_slot)), _ptr(y), _out_code(y.dtype), N, K,
                                        ctypes.c_void_p(status.data_ptr()) if status is not None else None,
                                        ctypes.c_void_p(_stream(stream)))
    _check(st, "nvfp4_moe_gemv_sdict")
    return y


def device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the library's device status bits."""
    v = ctypes.c_int32(0)
    st = library().nvfp4_device_status(ctypes.byref(v), ctypes.c_void_p(_stream(stream)))
    if st not in (0, 7):
        _check(st, "nvfp4_device_status")
    return int(v.value)


def set_wait_budget_ns(ns) -> None:
    """Budget of every device pipeline wait (None restores the default of 1 s)."""
    library().nvfp4_set_wait_budget_ns(ctypes.c_uint64((1 << 64) - 1 if ns is None else int(ns)))


def set_variant(variant: int) -> None:
    """0 = automatic kernel choice, 1 = byte-load kernel, 2 = streaming kernel with fp32 x."""
    library().nvfp4_set_variant(int(variant))


def fp32_fallbacks(stream=None) -> int:
    """CTAs that staged x in fp32 because block-scaled f16 could not hold it exactly
    (read and reset; synchronises the stream)."""
    v = library().nvfp4_fp32_fallbacks(ctypes.c_void_p(_stream(stream)))
    if v < 0:
        raise NVFP4Error(6, "nvfp4_fp32_fallbacks")
    return int(v)


def phase_trace(stream=None):
    """The phase trace of the last tile-kernel launches as an int64 tensor [16, 1024, 40]
    ([launch slot, CTA, word]; see nvfp4_phase_trace in the header), then cleared. None when
    the loaded library was built without tracing."""
    out = torch.zeros(16 * 1024 * 40, dtype=torch.int64)
    n = library().nvfp4_phase_trace(ctypes.c_void_p(out.data_ptr()), out.numel(), ctypes.c_void_p(_stream(stream)))
    if n < 0:
        raise NVFP4Error(6, "nvfp4_phase_trace")
    return out.view(16, 1024, 40) if n > 0 else None


def set_pdl(enable: bool) -> None:
    """Programmatic dependent launch between consecutive GEMVs (default on)."""
    library().nvfp4_set_pdl(int(bool(enable)))


KINDS = {"dense": 0, "gate_up": 1, "moe": 2, "moe_per_slot": 3, "gate_up_swiglu": 4, "dense_sdict": 5,
         "moe_sdict": 6, "moe_per_slot_sdict": 7, "ffn": 8}


def describe_plan(kind: str, M: int, N: int, K: int, T: int = 0, top_k: int = 0) -> str:
    """Launch the library would pick: kind is a key of KINDS; for the MoE kinds M is the number
    of experts (moe_per_slot: one x row per slot); for "ffn" N = H and K = I."""
    code = KINDS[kind]
    buf = ctypes.create_string_buffer(512)
    n = library().nvfp4_describe_plan(code, M, N, K, T, top_k, buf, 512)
    if n < 0:
        raise RuntimeError("describe_plan failed (no CUDA device?)")
    return buf.value.decode()


def describe_plan_host(kind: str, M: int, N: int, K: int, T: int = 0, top_k: int = 0, sm_count: int = 152,
                       smem_optin: int = 232448, smem_per_sm: int = 233472) -> str:
    """describe_plan for a described device (defaults: GB300), run on the host only: no GPU needed."""
    code = KINDS[kind]
    buf = ctypes.create_string_buffer(512)
    n = library().nvfp4_describe_plan_host(sm_count, smem_optin, smem_per_sm, code, M, N, K, T, top_k, buf, 512)
    if n < 0:
        raise ValueError("describe_plan_host: bad arguments")
    return buf.value.decode()
