"""Pins of the oracle's element / scale codecs (CPU only).

The formats are named on the block_scaled_quantization module page (NVFP4,
MXFP4, MXFP8) and defined by OCP MX v1.0.  Each encoder is checked against
something other than itself: an exact rational brute-force nearest search,
and PyTorch's float8 conversions (library routines) where their semantics
coincide.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import bf16_bits_to_f32

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _finite_bf16():
    v = bf16_bits_to_f32(ALL_BF16)
    return v[np.isfinite(v)]


def _brute_nearest(values, table_codes):
    """Exact brute force: among the (code, value) pairs pick the code whose
    value is nearest to v (Fractions), ties to the even code; the sign of v is
    then applied (|v| beyond the largest value keeps the largest)."""
    out = []
    for v in values:
        fv = Fraction(float(v))
        a = abs(fv)
        best = None
        for code, val in table_codes:
            d = abs(a - val)
            if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
                best = (d, code)
        out.append(best[1])
    return np.array(out, dtype=np.int64)


def _near_midpoints(mags, count=4):
    """FP32 values within a few ulps of every midpoint between adjacent
    magnitudes, of every magnitude, and just beyond the largest."""
    pts = []
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(len(mags) - 1)]
    for p in list(mids) + list(mags[1:]) + [mags[-1] * 1.0625]:
        x = np.float32(p)
        for _ in range(count):
            x = np.nextafter(x, np.float32(0))
        for _ in range(2 * count + 1):
            pts.append(x)
            x = np.nextafter(x, np.float32(np.inf))
    arr = np.array(pts, dtype=np.float32)
    return np.concatenate([arr, -arr])


# ---- decode tables -------------------------------------------------------

def test_e2m1_magnitudes_match_format_listing():
    # OCP MX v1.0 lists the FP4 E2M1 magnitudes explicitly.
    assert list(oracle.E2M1_MAGNITUDES) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(oracle.e2m1_decode(np.arange(8, 16))) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert np.signbit(oracle.e2m1_decode(8))


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_decode(np.arange(256))
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))
    assert oracle.E4M3_MAGNITUDES[-1] == 448.0 and len(oracle.E4M3_MAGNITUDES) == 127
    assert oracle.E4M3_MAGNITUDES[1] == 2.0 ** -9


def test_e8m0_decode_matches_torch():
    b = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e8m0_decode(np.arange(255)), ref)
    assert np.isnan(oracle.e8m0_decode(255))


# ---- encoders --------------------------------------------------------------

def test_e4m3_encode_matches_torch_in_range_all_bf16():
    v = _finite_bf16()
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_encode_matches_torch_random_fp32():
    rng = np.random.Generator(np.random.PCG64(11))
    u = rng.integers(0, 1 << 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    v = u.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    v = np.concatenate([v, (rng.standard_normal(200_000) * 50).astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_encode_saturates_beyond_448():
    v = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, 3.4e38], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), [0x7E] * len(v))
    np.testing.assert_array_equal(oracle.e4m3_encode(-v), [0xFE] * len(v))


def test_e4m3_encode_brute_force_near_midpoints():
    table = [(c, Fraction(float(m))) for c, m in enumerate(oracle.E4M3_MAGNITUDES)]
    v = _near_midpoints(oracle.E4M3_MAGNITUDES, count=2)
    ref = _brute_nearest(v, table) | np.where(np.signbit(v), 0x80, 0)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), ref)


def test_e2m1_encode_brute_force_all_bf16():
    v = _finite_bf16()
    table = [(c, Fraction(float(m))) for c, m in enumerate(oracle.E2M1_MAGNITUDES)]
    # brute force on the distinct magnitudes below the saturation point, then map
    small = np.unique(np.abs(v[np.abs(v) < 8.0]))
    ref_small = dict(zip(small.tolist(), _brute_nearest(small, table).tolist()))
    mag = np.abs(v)
    ref = np.array([ref_small[x] if x < 8.0 else 7 for x in mag.tolist()], dtype=np.int64)
    ref |= np.where(np.signbit(v), 0x8, 0)
    np.testing.assert_array_equal(oracle.e2m1_encode(v), ref)


def test_e2m1_encode_brute_force_near_midpoints():
    table = [(c, Fraction(float(m))) for c, m in enumerate(oracle.E2M1_MAGNITUDES)]
    v = _near_midpoints(oracle.E2M1_MAGNITUDES, count=4)
    ref = _brute_nearest(v, table) | np.where(np.signbit(v), 0x8, 0)
    np.testing.assert_array_equal(oracle.e2m1_encode(v), ref)


def test_encoders_keep_sign_of_zero_and_tiny():
    v = np.array([0.0, -0.0, 1e-45, -1e-45, -1e-30, 2.0 ** -11, -(2.0 ** -11)], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), [0, 0x80, 0, 0x80, 0x80, 0, 0x80])
    np.testing.assert_array_equal(oracle.e2m1_encode(v), [0, 8, 0, 8, 8, 0, 8])


def test_e8m0_ceil_exponent_closed_form():
    # powers of two and their FP32 neighbours, normal and subnormal
    ks = np.arange(-149, 128)
    p = np.ldexp(np.float32(1.0), ks).astype(np.float32)
    assert np.all(np.frexp(p)[0] == 0.5)
    np.testing.assert_array_equal(oracle.e8m0_ceil_exponent(p), ks)
    up = np.nextafter(p, np.float32(np.inf))
    np.testing.assert_array_equal(oracle.e8m0_ceil_exponent(up[ks < 127]), ks[ks < 127] + 1)
    # just below 2^k lies strictly inside (2^(k-1), 2^k) -- except below 2^-148,
    # where the next FP32 value down is 2^-149 itself
    down = np.nextafter(p[2:], np.float32(0))
    np.testing.assert_array_equal(oracle.e8m0_ceil_exponent(down), ks[2:])


def test_e8m0_ceil_exponent_exact_brute_force():
    rng = np.random.Generator(np.random.PCG64(5))
    u = rng.integers(1, 0x7F800000, size=5000, dtype=np.uint64).astype(np.uint32)
    s = u.view(np.float32)
    got = oracle.e8m0_ceil_exponent(s)
    for sv, e in zip(s.tolist(), got.tolist()):
        f = Fraction(sv)
        assert Fraction(2) ** e >= f > Fraction(2) ** (e - 1)
