"""Seeded synthetic inputs for the NVFP4 weight-only GEMV.

The test suite and the benchmark both draw their inputs from here. The module
encodes fp32 weights into the packed NVFP4 layout. It holds no decoding and no
product arithmetic, so it shares nothing with the CUDA kernels or the CPU oracle.
Both of those only consume the bytes produced here.

Quantisation recipe (two-level NVFP4, one block per 16 consecutive weights):

* ``g = amax(|W|) / (6 * 448)``, one FP32 scale per tensor (``g = 1`` if W is all zero).
* ``s_b = E4M3(amax_b / (6 * g))``. It is rounded to nearest-even and saturated to 448.
  The cast is torch's ``float8_e4m3fn`` conversion.
* ``q = E2M1(clamp(w / (E4M3(s_b) * g), -6, 6))``. It is rounded to the nearest of
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}, with ties to the even mantissa. ``q = 0`` where the
  decoded scale is 0.
* Codes are packed two per byte. Element ``2j`` of a row goes in the low nibble of
  byte ``j``.

Weights are ~N(0, 0.02) and activations ~N(0, 1) rounded to bf16. These are the
distributions of the attention, FFN, vocab-head and routed-expert workloads that
this library is measured on. Generation runs in fixed row chunks, so a given
``(seed, device)`` always yields the same bytes. CPU and CUDA generators give
different (but each reproducible) streams.
"""
from __future__ import annotations

import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0
_CHUNK_ELEMS = 1 << 24  # rows are generated in chunks of about this many elements


def _encode_e2m1(v: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (ties to even mantissa) of values already in [-6, 6]."""
    a = v.abs()
    mag = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8)
           + (a > 1.25).to(torch.uint8) + (a >= 1.75).to(torch.uint8)
           + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
           + (a > 5.0).to(torch.uint8))
    sign = (v < 0).to(torch.uint8) << 3
    return mag | sign


def quantize(w: torch.Tensor, g: float | None = None):
    """Encode fp32 ``w [N, K]`` (K % 16 == 0) as NVFP4.

    Returns ``(packed u8 [N, K/2], scales u8 [N, K/16], g)`` on w's device.
    Pass ``g`` to quantise a row chunk of a larger tensor with that tensor's scale.
    """
    N, K = w.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    w = w.to(torch.float32)
    if g is None:
        amax = float(w.abs().max()) if w.numel() else 0.0
        g = amax / (6.0 * E4M3_MAX) if amax > 0 else 1.0
    g = float(torch.tensor(g, dtype=torch.float32))  # the FP32 value the kernels get
    blocks = w.reshape(N, K // 16, 16)
    bamax = blocks.abs().amax(dim=-1)
    sf = (bamax / (6.0 * g)).clamp(max=E4M3_MAX).to(torch.float8_e4m3fn)
    scales = sf.view(torch.uint8)
    denom = sf.to(torch.float32) * g
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    q = torch.where((denom > 0)[..., None], blocks / safe[..., None], torch.zeros_like(blocks))
    codes = _encode_e2m1(q.clamp(-E2M1_MAX, E2M1_MAX)).reshape(N, K)
    packed = codes[:, 0::2] | (codes[:, 1::2] << 4)
    return packed.contiguous(), scales.contiguous(), g


def _gen(seed: int, device) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(int(seed))


def random_weight(N: int, K: int, seed: int, device="cpu", std: float = 0.02):
    """A ~N(0, std) [N, K] weight quantised to NVFP4: ``(packed, scales, g)``.

    Two passes over the same seeded stream: the first finds amax(|W|), the second
    quantises chunk by chunk, so memory stays bounded for vocab-sized tensors.
    """
    rows = max(1, _CHUNK_ELEMS // max(K, 1))
    amax = 0.0
    gen = _gen(seed, device)
    for r0 in range(0, N, rows):
        n = min(rows, N - r0)
        amax = max(amax, float((torch.randn(n, K, generator=gen, device=device) * std).abs().max()))
    g = amax / (6.0 * E4M3_MAX) if amax > 0 else 1.0
    packed = torch.empty(N, K // 2, dtype=torch.uint8, device=device)
    scales = torch.empty(N, K // 16, dtype=torch.uint8, device=device)
    gen = _gen(seed, device)
    for r0 in range(0, N, rows):
        n = min(rows, N - r0)
        w = torch.randn(n, K, generator=gen, device=device) * std
        p, s, g = quantize(w, g)
        packed[r0:r0 + n] = p
        scales[r0:r0 + n] = s
    return packed, scales, g


def _quantize_with_codes(w: torch.Tensor, g: float, codes: torch.Tensor):
    """quantize() with every block scale drawn from ``codes`` (u8 E4M3 codes, increasing in
    value): the smallest code whose value is >= amax_b / (6 g), else the largest code."""
    N, K = w.shape
    blocks = w.to(torch.float32).reshape(N, K // 16, 16)
    need = blocks.abs().amax(dim=-1) / (6.0 * g)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float32)
    pick = torch.searchsorted(vals, need.contiguous()).clamp(max=codes.numel() - 1)
    scales = codes[pick]
    denom = scales.view(torch.float8_e4m3fn).to(torch.float32) * g
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    q = torch.where((denom > 0)[..., None], blocks / safe[..., None], torch.zeros_like(blocks))
    c = _encode_e2m1(q.clamp(-E2M1_MAX, E2M1_MAX)).reshape(N, K)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous(), scales.contiguous()


def random_weight_sdict(N: int, K: int, seed: int, device="cpu", std: float = 0.02, max_codes: int = 32):
    """random_weight() whose block scales take at most ``max_codes`` distinct E4M3 codes, so that
    the tensor has a scale-dictionary form. When the plain recipe gives more, the most frequent
    codes are kept and every block takes the smallest kept code that still covers its amax
    (no E2M1 clipping), the codes requantised with it."""
    packed, scales, g = random_weight(N, K, seed, device, std)
    vals, counts = torch.unique(scales, return_counts=True)
    if vals.numel() <= max_codes:
        return packed, scales, g
    keep = vals[counts.argsort(descending=True)[:max_codes]]
    keep = keep[keep.view(torch.float8_e4m3fn).to(torch.float32).argsort()]
    rows = max(1, _CHUNK_ELEMS // max(K, 1))
    gen = _gen(seed, device)  # the stream random_weight quantised, drawn again chunk by chunk
    for r0 in range(0, N, rows):
        n = min(rows, N - r0)
        w = torch.randn(n, K, generator=gen, device=device) * std
        packed[r0:r0 + n], scales[r0:r0 + n] = _quantize_with_codes(w, g, keep)
    return packed, scales, g


def sdict_problem(N: int, K: int, M: int, seed: int, device="cpu"):
    """A dense problem whose weight has at most 32 scale codes: dict(w, s, g, x), s plain."""
    w, s, g = random_weight_sdict(N, K, seed * 2 + 1, device)
    return {"w": w, "s": s, "g": g, "x": random_x(M, K, seed * 2 + 2, device), "N": N, "K": K, "M": M}


def sdict_pack(ind: torch.Tensor, N: int, K: int) -> torch.Tensor:
    """Index plane of a scale-dictionary tensor from its block indices ind [N, K/16] (0..31):
    one 160-byte record per 16-row tile r and 256-column segment c at byte (r * K/256 + c) * 160,
    the index of (row 16r + i, block 16c + j) at bits 5q .. 5q + 4 (q = 16i + j, least significant
    first; bit p of a record is bit p % 8 of byte p / 8). The 8 indices q = 8p .. 8p + 7 fill
    bytes 5p .. 5p + 4. Returns uint8 [((N + 15) // 16) * (K // 256) * 160] on the CPU."""
    segs, tiles = K // 256, (N + 15) // 16
    full = torch.zeros(tiles * 16, K // 16, dtype=torch.int64)
    full[:N] = ind.to("cpu", torch.int64)
    rec = full.reshape(tiles, 16, segs, 16).permute(0, 2, 1, 3).reshape(tiles, segs, 32, 8)
    v = torch.zeros(rec.shape[:3], dtype=torch.int64)
    for k in range(8):
        v |= rec[..., k] << (5 * k)
    out = torch.stack([(v >> (8 * m)) & 0xFF for m in range(5)], dim=-1).to(torch.uint8)
    return out.reshape(-1)


def sdict_form(s: torch.Tensor):
    """Dictionary form of plain block scales s [N, K/16] with at most 32 distinct codes: the
    table holds the codes in increasing byte order (its tail repeats the last one), each block
    its code's position. Returns (index plane, table [32]) as uint8 tensors on s's device.
    For s [E, N, K/16] (one dictionary per expert) returns ([E, plane], [E, 32])."""
    if s.dim() == 3:
        forms = [sdict_form(s[e]) for e in range(s.shape[0])]
        return torch.stack([f[0] for f in forms]), torch.stack([f[1] for f in forms])
    codes = torch.unique(s.to("cpu"))
    if not 0 < codes.numel() <= 32:
        raise ValueError(f"{codes.numel()} distinct scale codes: no dictionary form")
    table = torch.cat([codes, codes[-1:].repeat(32 - codes.numel())]).to(torch.uint8)
    ind = torch.searchsorted(codes, s.to("cpu").contiguous())
    return sdict_pack(ind, s.shape[0], s.shape[1] * 16).to(s.device), table.to(s.device)


def random_x(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 activations ~N(0, 1), shape [M, K]."""
    return torch.randn(M, K, generator=_gen(seed, device), device=device).to(torch.bfloat16)


def dense_problem(N: int, K: int, M: int, seed: int, device="cpu"):
    """One dense problem: dict(w, s, g, x). The weight and x use seeds derived from ``seed``."""
    w, s, g = random_weight(N, K, seed * 2 + 1, device)
    x = random_x(M, K, seed * 2 + 2, device)
    return {"w": w, "s": s, "g": g, "x": x, "N": N, "K": K, "M": M}


def gate_up_problem(N: int, K: int, M: int, seed: int, device="cpu"):
    """Gate and up weights (each [N, K]) with their own global scales, one x [M, K]."""
    wg, sg, gg = random_weight(N, K, seed * 3 + 1, device)
    wu, su, gu = random_weight(N, K, seed * 3 + 2, device)
    x = random_x(M, K, seed * 3 + 3, device)
    return {"wg": wg, "sg": sg, "gg": gg, "wu": wu, "su": su, "gu": gu, "x": x,
            "N": N, "K": K, "M": M}


def ffn_problem(H: int, I: int, M: int, seed: int, device="cpu"):
    """An FFN block: gate and up weights [I, H], down weight [H, I], each with its own global
    scale, and x [M, H]."""
    wg, sg, gg = random_weight(I, H, seed * 4 + 1, device)
    wu, su, gu = random_weight(I, H, seed * 4 + 2, device)
    wd, sd, gd = random_weight(H, I, seed * 4 + 3, device)
    x = random_x(M, H, seed * 4 + 4, device)
    return {"wg": wg, "sg": sg, "gg": gg, "wu": wu, "su": su, "gu": gu, "wd": wd, "sd": sd, "gd": gd, "x": x,
            "H": H, "I": I, "M": M}


def routing(T: int, top_k: int, E: int, seed: int) -> torch.Tensor:
    """Expert ids [T * top_k] int32, token-major. Each token draws top_k distinct experts
    uniformly without replacement (a seeded permutation, first top_k entries)."""
    gen = _gen(seed, "cpu")
    ids = [torch.randperm(E, generator=gen)[:top_k] for _ in range(T)]
    return torch.cat(ids).to(torch.int32) if ids else torch.empty(0, dtype=torch.int32)


def moe_problem(E: int, N: int, K: int, T: int, top_k: int, x_per_slot: bool, seed: int,
                device="cpu", fill: str = "routed", ids=None, max_codes: int | None = None):
    """Routed-expert problem: w [E, N, K/2], s [E, N, K/16], gs [E] f32, ids, x.

    Expert e's weight comes from seed ``seed * 1000 + e``. ``fill="routed"``
    generates only the experts that ``ids`` names. The others keep zero bytes
    (code 0, scale 0) and a global scale of 1. That is enough for anything that reads only the routed
    slabs, and it keeps CPU generation fast. ``fill="all"`` generates every expert. ``ids``
    (T * top_k ints) replaces the seeded routing when given. ``max_codes`` limits each expert's
    block scales to that many distinct codes (random_weight_sdict).
    """
    ids = routing(T, top_k, E, seed) if ids is None else torch.as_tensor(ids, dtype=torch.int32).reshape(-1).cpu()
    assert ids.numel() == T * top_k
    w = torch.zeros(E, N, K // 2, dtype=torch.uint8, device=device)
    s = torch.zeros(E, N, K // 16, dtype=torch.uint8, device=device)
    gs = torch.ones(E, dtype=torch.float32)
    experts = range(E) if fill == "all" else sorted(set(int(e) for e in ids.tolist() if 0 <= int(e) < E))
    for e in experts:
        if max_codes is None:
            we, se, ge = random_weight(N, K, seed * 1000 + e, device)
        else:
            we, se, ge = random_weight_sdict(N, K, seed * 1000 + e, device, max_codes=max_codes)
        w[e], s[e], gs[e] = we, se, ge
    rows = T * top_k if x_per_slot else T
    x = random_x(rows, K, seed * 1000 + E + 7, device)
    return {"w": w, "s": s, "gs": gs.to(device), "ids": ids.to(device), "x": x, "E": E,
            "N": N, "K": K, "T": T, "top_k": top_k, "x_per_slot": bool(x_per_slot)}


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
