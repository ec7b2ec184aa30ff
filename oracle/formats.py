"""Number formats of the index-K cache, written from their definitions.

bf16: IEEE-754 binary32 with the low 16 bits dropped (1 sign, 8 exponent,
7 fraction bits). Rounding from binary32 is round-to-nearest-even.

E4M3 (OCP 8-bit Floating Point Specification, "E4M3" format): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits. Normal values
(-1)^s * 2^(e-7) * (1 + m/8) for e in 1..15 except the all-ones pattern
S.1111.111, which is NaN; subnormals (-1)^s * 2^-6 * m/8 for e = 0. There are
no infinities; the largest finite magnitude is 448 (S.1111.110).

The fp8 index key is 128 such bytes plus one fp32 scale per token ("The Moment
of Validation", section "Input Knowledge Required to Understand This Message":
132 bytes per token, a shared scale factor per group).

E2M1 (OCP Microscaling Formats (MX) Specification v1.0, section 5.3.3, the
FP4 element type): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit.
Normal values (-1)^s * 2^(e-1) * (1 + m/2) for e in 1..3, subnormals
(-1)^s * m/2 for e = 0: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. There are no
infinities and no NaN. The fp4 index key of this library is 128 such codes
(two per byte, the even dimension in the low nibble) plus one fp32 scale per
token: the fp8 key with its element type narrowed ("The Fused Kernel
Decision", section "The Message: A Blueprint for Kernel Modification", names
an fp4 variant for more aggressive compression and gives no layout; this is
the plainest reading of it).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest, ties to even). Returns bit patterns.

    The kept part is the top 16 bits; the dropped part d (low 16 bits) decides:
    d > 0x8000 rounds up, d < 0x8000 rounds down, d == 0x8000 rounds to the
    even kept pattern. NaNs map to a quiet NaN.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    hi = (u >> np.uint32(16)).astype(np.uint32)
    lo = u & np.uint32(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint32(1)) == 1))
    r = hi + up.astype(np.uint32)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(nan, (hi | np.uint32(0x40)) & np.uint32(0xFFFF), r)
    return r.astype(np.uint16)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 codes (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** -9                       # 2^-6 * m/8
    nrm = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32))
    v = np.where(e == 0, sub, nrm)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def f32_to_e4m3_satfinite(x: np.ndarray) -> np.ndarray:
    """binary32 -> E4M3 code, round to nearest even, saturating to +-448.

    For |x| < 448 the result is the representable value nearest |x|: the
    spacing of representable values in the binade [2^E, 2^(E+1)) is 2^(E-3),
    and below 2^-6 (the subnormal range) it is 2^-9. |x| is divided by that
    spacing (exact: a power of two), rounded to an integer with ties to even,
    and multiplied back. Magnitudes >= 448 give 448. The sign is kept (so -0
    gives 0x80). NaN gives 0x7F.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    sign = np.signbit(x)
    _, ex = np.frexp(a)                        # a = f * 2^ex, f in [0.5, 1)
    E = np.maximum(ex.astype(np.int64) - 1, -6)
    E = np.where(a == 0.0, -6, E)
    quantum = np.ldexp(1.0, (E - 3).astype(np.int32))
    v = np.rint(a / quantum) * quantum         # np.rint: ties to even
    v = np.minimum(v, E4M3_MAX)
    v = np.where(a >= E4M3_MAX, E4M3_MAX, v)
    # encode v (exactly representable now)
    _, ev = np.frexp(v)
    Ev = ev.astype(np.int64) - 1
    is_sub = (v < 2.0 ** -6)
    m_sub = np.rint(v / 2.0 ** -9).astype(np.int64)
    e_nrm = Ev + 7
    m_nrm = np.rint((v / np.ldexp(1.0, Ev.astype(np.int32)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(is_sub, m_sub, (e_nrm << 3) | m_nrm)
    code = np.where(sign, code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def e2m1_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of E2M1 codes (the low 4 bits of each entry)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    s = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    sub = m * 0.5                              # 2^0 * m/2
    nrm = np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int32))
    return s * np.where(e == 0, sub, nrm)


def f32_to_e2m1_satfinite(x: np.ndarray) -> np.ndarray:
    """binary32 -> E2M1 code (0..15), round to nearest even, saturating to +-6.

    The spacing of representable magnitudes is 0.5 below 2 (the subnormal
    step and the step of the binade [1, 2)), 1 in [2, 4) and 2 in [4, 6]:
    |x| is divided by its spacing, rounded to an integer with ties to even,
    and multiplied back; magnitudes >= 6 give 6. The sign is kept (-0 gives
    code 8).
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.abs(x)
    sign = np.signbit(x)
    quantum = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    v = np.minimum(np.rint(a / quantum) * quantum, E2M1_MAX)
    # encode v: 0, 0.5 -> 0, 1; then 1 + 2(e-1) + m for the normal values
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    code = np.vectorize(lambda t: table[float(t)], otypes=[np.int64])(v) if v.size else v.astype(np.int64)
    code = np.where(sign, code | 0x8, code)
    return code.astype(np.uint8)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Pack codes [..., 2n] two per byte: element 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_e2m1: codes [..., 2n] from bytes [..., n]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
