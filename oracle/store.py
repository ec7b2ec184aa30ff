"""Oracle for the index-key store: RMSNorm + RoPE + quantise + paged write.

What the store computes ("The Moment of Validation", section "Input
Knowledge Required to Understand This Message": the fused kernel normalises,
applies RoPE and stores each index key in one pass; "The Fused Kernel
Decision", section "The Message": a 64-token paged layout in which a token
maps to a page and an offset inside it):

  y    = RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma       (128 dims)
  y'   = RoPE(y, pos), dims i and i+64 rotated by pos * theta^(-2i/128)
  bf16 : store round(y') as 128 bf16 values                   (256 B/token)
  fp8  : scale = max|y'| / 448, store e4m3(y' / scale) (128 B) and the fp32
         scale (4 B)                                          (132 B/token)
  fp4  : scale = max|y'| / 6, store e2m1(y' / scale) two codes per byte
         (64 B) and the fp32 scale (4 B)                      (68 B/token)
         (the pages name an fp4 variant but give no layout: this reading
         is the fp8 key with e2m1 elements, see oracle.formats)

The bytes are decided by floating point, so the oracle computes them in the
precision the kernel uses (fp32) with one fixed order of operations, which is
the definition the stored bytes are compared against:

  * sum of squares: 16 partial sums over consecutive groups of 8 dims,
    each accumulated in dim order; then the partials are added pairwise,
    (g, g+8), then (g, g+4), (g, g+2), (g, g+1);
  * mean = sum * (1/128) (exact); r = 1 / sqrt(mean + eps), each operation
    rounded to nearest;
  * y_d = (x_d * r) * gamma_d;
  * RoPE, with c = cos(pos*f_i), s = sin(pos*f_i), f_i = theta^(-2i/128)
    evaluated in double by the host C library and rounded once to fp32:
        y'_i      = y_i * c - y_{i+64} * s
        y'_{i+64} = y_{i+64} * c + y_i * s
    every product and sum rounded separately (no fused multiply-add);
  * fp8: amax = max(max_d |y'_d|, 1e-4); scale = amax / 448;
    inv = 1 / scale; code_d = e4m3_satfinite(y'_d * inv).
  * fp4: the same with 6 for 448 and e2m1_satfinite for e4m3_satfinite.

The 1e-4 floor on amax is this library's reading for an all-zero key (the
pages do not say); it keeps the scale positive, which the scorer relies on.

Optional Hadamard rotation ("The Moment of Validation", section "Input
Knowledge Required to Understand This Message": the fused kernel applies a
Hadamard transform between RoPE and the store; "The Fused Kernel Decision",
section "Assumptions and Their Validity": queries and keys must come out in
the same order). The pages fix neither the normalisation nor the order; the
reading taken here is the unnormalised 128-point Walsh-Hadamard transform in
natural (Sylvester) order, applied to y' before quantisation:
    stages h = 1, 2, 4, ..., 64: every pair (i, i+h) with i & h == 0
    becomes (a + b, a - b), each sum rounded to fp32.
Its matrix H has entries +-1 and H H^T = 128 I, so a query rotated the same
way gives (H q) . (H k) = 128 (q . k); the scorer divides by 128 (exact).

Cache layouts (per page of 64 tokens):
  bf16 : [64][128] bf16                         16384 bytes
  fp8  : [64][128] e4m3, then [64] fp32 scales   8448 bytes
  fp4  : [64][64] e2m1 pairs, then [64] fp32 scales  4352 bytes
"""
from __future__ import annotations

import math

import numpy as np

from . import formats as F

D = 128
HALF = 64
PAGE = 64
FMT_BF16 = 0
FMT_FP8 = 1
FMT_FP4 = 2
PAGE_BYTES = {FMT_BF16: PAGE * D * 2, FMT_FP8: PAGE * D + PAGE * 4, FMT_FP4: PAGE * D // 2 + PAGE * 4}
TOKEN_BYTES = {FMT_BF16: D * 2, FMT_FP8: D + 4, FMT_FP4: D // 2 + 4}
CODE_BYTES = {FMT_FP8: D, FMT_FP4: D // 2}  # per token, before the page's scales
AMAX_FLOOR = np.float32(1e-4)


def rope_cos_sin(theta: float, positions: np.ndarray):
    """fp32 cos/sin of pos * theta^(-2i/128) for i < 64, from double libm."""
    positions = np.asarray(positions, dtype=np.int64)
    uniq, inv = np.unique(positions, return_inverse=True)
    th = float(np.float32(theta))            # theta is an fp32 parameter of the store
    freqs = [math.pow(th, -(2.0 * i) / D) for i in range(HALF)]
    cu = np.empty((len(uniq), HALF), dtype=np.float32)
    su = np.empty((len(uniq), HALF), dtype=np.float32)
    for r, p in enumerate(uniq.tolist()):
        cu[r] = [math.cos(p * f) for f in freqs]
        su[r] = [math.sin(p * f) for f in freqs]
    return cu[inv], su[inv]


def sum_squares_f32(x: np.ndarray) -> np.ndarray:
    """fp32 sum of squares of rows [T,128] in the fixed order stated above:
    16 partials over dims 8g..8g+7 in dim order, then pairwise (g, g+8),
    (g, g+4), (g, g+2), (g, g+1)."""
    x = np.asarray(x, dtype=np.float32)
    T = x.shape[0]
    sq = (x * x).reshape(T, 16, 8)            # exact: x has <= 8 significant bits
    p = sq[:, :, 0].copy()
    for j in range(1, 8):
        p = p + sq[:, :, j]
    t = p[:, :8] + p[:, 8:]
    t = t[:, :4] + t[:, 4:]
    t = t[:, :2] + t[:, 2:]
    return t[:, 0] + t[:, 1]


def rmsnorm_f32(x: np.ndarray, eps: float, gamma: np.ndarray | None = None) -> np.ndarray:
    """RMSNorm of fp32 rows [T,128] in the fixed fp32 order stated above."""
    x = np.asarray(x, dtype=np.float32)
    ss = sum_squares_f32(x)
    ms = ss * np.float32(1.0 / 128.0)
    r = np.float32(1.0) / np.sqrt(ms + np.float32(eps))
    y = x * r[:, None]
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float32)[None, :]
    return y


def rope_f32(y: np.ndarray, c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Half-split RoPE in fp32, each operation rounded separately."""
    a = y[:, :HALF]
    b = y[:, HALF:]
    out = np.empty_like(y)
    out[:, :HALF] = a * c - b * s
    out[:, HALF:] = b * c + a * s
    return out


def wht_f32(y: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of fp32 rows [T,128], natural
    order, butterfly stages h = 1, 2, ..., 64 with fp32 sums."""
    y = np.array(y, dtype=np.float32, copy=True)
    T = y.shape[0]
    h = 1
    while h < D:
        v = y.reshape(T, D // (2 * h), 2, h)
        a = v[:, :, 0, :].copy()
        b = v[:, :, 1, :].copy()
        v[:, :, 0, :] = a + b
        v[:, :, 1, :] = a - b
        h *= 2
    return y


def normalize_rotate(k_raw_bits: np.ndarray, pos: np.ndarray, theta: float, eps: float,
                     gamma_bits: np.ndarray | None = None, hadamard: bool = False) -> np.ndarray:
    """fp32 y' (then H y' when hadamard) for bf16 raw keys [T,128] at
    positions pos [T]."""
    x = F.bf16_to_f64(k_raw_bits).astype(np.float32)
    gamma = None if gamma_bits is None else F.bf16_to_f64(gamma_bits).astype(np.float32)
    y = rmsnorm_f32(x, eps, gamma)
    c, s = rope_cos_sin(theta, pos)
    yr = rope_f32(y, c, s)
    return wht_f32(yr) if hadamard else yr


def quantize_fp8(yr: np.ndarray):
    """Per-token amax scale and e4m3 codes of fp32 rows."""
    amax = np.maximum(np.max(np.abs(yr), axis=1), AMAX_FLOOR).astype(np.float32)
    scale = (amax / np.float32(F.E4M3_MAX)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    codes = F.f32_to_e4m3_satfinite(yr * inv[:, None])
    return codes, scale


def quantize_fp4(yr: np.ndarray):
    """Per-token amax scale and packed e2m1 codes [T,64] of fp32 rows."""
    amax = np.maximum(np.max(np.abs(yr), axis=1), AMAX_FLOOR).astype(np.float32)
    scale = (amax / np.float32(F.E2M1_MAX)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    codes = F.f32_to_e2m1_satfinite(yr * inv[:, None])
    return F.pack_e2m1(codes), scale


def new_cache(num_pages: int, fmt: int) -> np.ndarray:
    return np.zeros(num_pages * PAGE_BYTES[fmt], dtype=np.uint8)


def slots(pos: np.ndarray, seq: np.ndarray, page_table: np.ndarray, num_pages: int):
    """(page, offset) of each token: page_table[seq][pos // 64], pos % 64."""
    pos = np.asarray(pos, dtype=np.int64)
    seq = np.asarray(seq, dtype=np.int64)
    page = np.asarray(page_table, dtype=np.int64)[seq, pos // PAGE]
    if np.any((page < 0) | (page >= num_pages)):
        raise ValueError("page id out of range")
    return page, pos % PAGE


def _views(cache: np.ndarray, fmt: int):
    """Per-page views of the cache bytes: bf16 -> [pages, 64, 256] bytes;
    fp8 -> ([pages, 64, 128] codes, [pages, 64] fp32 scales); fp4 ->
    ([pages, 64, 64] packed codes, [pages, 64] fp32 scales)."""
    pb = PAGE_BYTES[fmt]
    pages = cache.reshape(-1, pb)
    if fmt == FMT_BF16:
        return pages.reshape(-1, PAGE, 2 * D), None
    cb = CODE_BYTES[fmt]
    data = pages[:, :PAGE * cb].reshape(-1, PAGE, cb)
    scales = pages[:, PAGE * cb:].view("<f4")
    return data, scales


def store(cache: np.ndarray, fmt: int, k_raw_bits, pos, seq, page_table, num_pages: int,
          theta: float = 10000.0, eps: float = 1e-6, gamma_bits=None, hadamard: bool = False) -> None:
    """Write the tokens' index keys into the byte image of the paged cache."""
    if len(pos) == 0:
        return
    yr = normalize_rotate(k_raw_bits, pos, theta, eps, gamma_bits, hadamard)
    page, off = slots(pos, seq, page_table, num_pages)
    data, scales = _views(cache, fmt)
    if fmt == FMT_BF16:
        data[page, off] = F.f32_to_bf16(yr).view(np.uint8).reshape(-1, 2 * D)
    else:
        codes, scale = quantize_fp8(yr) if fmt == FMT_FP8 else quantize_fp4(yr)
        data[page, off] = codes
        scales[page, off] = scale


def read_keys(cache: np.ndarray, fmt: int, page_table_row: np.ndarray, n: int) -> np.ndarray:
    """Exact float64 values of the stored keys at positions 0..n-1 of one
    sequence (fp8 / fp4: the e4m3 / e2m1 value times the token's scale,
    exact in double)."""
    if n == 0:
        return np.zeros((0, D))
    pos = np.arange(n, dtype=np.int64)
    page = np.asarray(page_table_row, dtype=np.int64)[pos // PAGE]
    off = pos % PAGE
    data, scales = _views(cache, fmt)
    if fmt == FMT_BF16:
        return F.bf16_to_f64(np.ascontiguousarray(data[page, off]).view(np.uint16))
    codes = data[page, off]
    vals = F.e4m3_to_f64(codes) if fmt == FMT_FP8 else F.e2m1_to_f64(F.unpack_e2m1(codes))
    return vals * scales[page, off].astype(np.float64)[:, None]
