"""Pins for the oracle's number formats (bf16, OCP E4M3, OCP MX E2M1),
against the formats' definitions, hand-written tables from the OCP FP8 and
MX specifications, and torch's own CPU conversions as an independent library
routine."""
import os

import numpy as np
import pytest

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_codes():
    rows = []
    with open(os.path.join(GOLD, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, c = line.split()[:2]
            rows.append((float(v), int(c, 16)))
    return rows


def test_e4m3_golden_table():
    rows = _golden_codes()
    vals = np.array([v for v, _ in rows], dtype=np.float32)
    want = np.array([c for _, c in rows], dtype=np.uint8)
    got = F.f32_to_e4m3_satfinite(vals)
    assert got.tolist() == want.tolist()


def test_e4m3_all_codes_roundtrip():
    codes = np.arange(256, dtype=np.uint8)
    v = F.e4m3_to_f64(codes)
    nan = np.isnan(v)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    enc = F.f32_to_e4m3_satfinite(v[~nan].astype(np.float32))
    assert np.array_equal(enc, codes[~nan])


def test_e4m3_decode_by_formula():
    # value = (-1)^s 2^(e-7) (1 + m/8), subnormal 2^-6 m/8, enumerated by hand loops
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = (2.0 ** -6) * (m / 8.0) if e == 0 else (2.0 ** (e - 7)) * (1 + m / 8.0)
        v = -v if s else v
        assert F.e4m3_to_f64(np.array([c], np.uint8))[0] == v


def test_e4m3_midpoints_round_to_even():
    vals = np.sort(np.unique(F.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = (vals[:-1] + vals[1:]) / 2          # exact in fp32 (<= 5 significant bits)
    got = F.e4m3_to_f64(F.f32_to_e4m3_satfinite(mids.astype(np.float32)))
    lo_code = F.f32_to_e4m3_satfinite(vals[:-1].astype(np.float32))
    even_is_lo = (lo_code & 1) == 0
    want = np.where(even_is_lo, vals[:-1], vals[1:])
    assert np.array_equal(got, want)


def test_e4m3_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) < 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(t, F.f32_to_e4m3_satfinite(x))


def test_e4m3_nearest_bruteforce():
    # the code whose value is nearest |x| (ties: even code), by exhaustive search
    table = F.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    rng = np.random.default_rng(2)
    x = np.abs(rng.standard_normal(3000) * np.exp(rng.uniform(-9, 6, 3000))).astype(np.float32)
    got = F.f32_to_e4m3_satfinite(x)
    for xi, gi in zip(x.astype(np.float64), got):
        if xi >= 448:
            assert gi == 0x7E
            continue
        d = np.abs(table - xi)
        best = np.nonzero(d == d.min())[0]
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert gi == want


def test_bf16_rne_matches_torch_and_definition():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    # add exact ties: low 16 bits == 0x8000
    u = x.view(np.uint32).copy()
    u[:1000] = (u[:1000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = u.view(np.float32)
    b = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, F.f32_to_bf16(x))
    # ties go to the even pattern
    t = F.f32_to_bf16(x[:1000])
    assert np.all((t & 1) == 0)


def test_bf16_decode_exact():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_to_f64(bits)
    fin = np.isfinite(v)
    assert np.array_equal(F.f32_to_bf16(v[fin].astype(np.float32)), bits[fin])


def _golden_e2m1():
    rows = []
    with open(os.path.join(GOLD, "e2m1_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, c = line.split()[:2]
            rows.append((float(v), int(c, 16)))
    return rows


def test_e2m1_golden_table():
    rows = _golden_e2m1()
    vals = np.array([v for v, _ in rows], dtype=np.float32)
    want = [c for _, c in rows]
    assert F.f32_to_e2m1_satfinite(vals).tolist() == want


def test_e2m1_decode_by_formula():
    # value = (-1)^s 2^(e-1) (1 + m/2), subnormal m/2, enumerated by hand loops
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = F.e2m1_to_f64(np.arange(16, dtype=np.uint8))
    assert got[:8].tolist() == want
    assert got[8:].tolist() == [-v for v in want]
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        v = m / 2.0 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2.0)
        assert got[c] == (-v if s else v)


def test_e2m1_all_codes_roundtrip():
    codes = np.arange(16, dtype=np.uint8)
    v = F.e2m1_to_f64(codes)
    assert np.array_equal(F.f32_to_e2m1_satfinite(v.astype(np.float32)), codes)


def test_e2m1_nearest_bruteforce():
    # the code whose value is nearest |x| (ties: even code), by exhaustive search
    table = F.e2m1_to_f64(np.arange(8, dtype=np.uint8))
    rng = np.random.default_rng(4)
    x = np.abs(rng.standard_normal(4000) * np.exp(rng.uniform(-3, 3, 4000))).astype(np.float32)
    x = np.concatenate([x, (np.arange(0, 29) / 4.0).astype(np.float32)])  # every quarter to 7
    got = F.f32_to_e2m1_satfinite(x)
    for xi, gi in zip(x.astype(np.float64), got):
        if xi >= 6:
            assert gi == 0x7
            continue
        d = np.abs(table - xi)
        best = np.nonzero(d == d.min())[0]
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert gi == want


def test_e2m1_pack_nibble_order():
    # element 2i sits in the low nibble of byte i
    codes = np.array([[0x1, 0x7, 0x8, 0xF, 0x2, 0x0]], np.uint8)
    p = F.pack_e2m1(codes)
    assert p.tolist() == [[0x71, 0xF8, 0x02]]
    assert np.array_equal(F.unpack_e2m1(p), codes)
