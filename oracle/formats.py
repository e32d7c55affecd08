"""Element and scale codecs (oracle; test infrastructure only).

The pages name the formats ("NVFP4, MXFP4, and MXFP8", block_scaled_quantization
module index) but never define them.  The definitions below are the OCP
Microscaling v1.0 ones:

* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no Inf/NaN.
* E4M3 (FN): 1 sign, 4 exponent (bias 7), 3 mantissa bits; 0x7F/0xFF NaN,
  no Inf, largest finite 448.
* E8M0: 8-bit biased exponent, value 2^(b-127), 0xFF NaN.

Encoding (FP32 -> E2M1 / E4M3) is "nearest representable magnitude, ties to
the even code, saturate beyond the largest finite magnitude, keep the sign
bit".  The nearest search compares the two bracketing magnitudes in float64.
That decision is exact: float64 subtraction is monotone, so it cannot invert
an order, and it cannot merge two different distances into a false tie
because, whenever both candidates are close to v, v - m is exactly
representable in float64 (an FP32 v and a code with at most 4 significant
bits span far fewer than 53 bits).
"""
from __future__ import annotations

import numpy as np


def _e2m1_value(code: int) -> float:
    e, m = (code >> 1) & 0x3, code & 0x1
    mag = 0.5 * m if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if code & 0x8 else mag


def _e4m3_value(code: int) -> float:
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if code & 0x80 else mag


# magnitudes of the non-negative codes, indexed by code (increasing)
E2M1_MAGNITUDES = np.array([_e2m1_value(c) for c in range(8)], dtype=np.float64)
E4M3_MAGNITUDES = np.array([_e4m3_value(c) for c in range(0x7F)], dtype=np.float64)
_E2M1_ALL = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
_E4M3_ALL = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 code (low 4 bits) -> float64 value."""
    return _E2M1_ALL[np.asarray(codes, dtype=np.int64) & 0xF]


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte -> float64 value (NaN for 0x7F / 0xFF)."""
    return _E4M3_ALL[np.asarray(codes, dtype=np.int64) & 0xFF]


def e8m0_decode(codes) -> np.ndarray:
    """E8M0 byte -> float64 value 2^(b-127) (NaN for 0xFF)."""
    b = np.asarray(codes, dtype=np.int64)
    return np.where(b == 0xFF, np.nan, np.ldexp(1.0, b - 127))


def _encode_nearest(v, magnitudes: np.ndarray, sign_bit: int) -> np.ndarray:
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    last = len(magnitudes) - 1
    hi = np.minimum(np.searchsorted(magnitudes, a, side="left"), last)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - magnitudes[lo]
    d_hi = magnitudes[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a >= magnitudes[last], last, code)       # saturate
    code = code | np.where(np.signbit(v), sign_bit, 0)
    return code.astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """FP32 -> E2M1 code (0..15): nearest, ties to even, satfinite, sign kept."""
    return _encode_nearest(v, E2M1_MAGNITUDES, 0x8)


def e4m3_encode(v) -> np.ndarray:
    """FP32 -> E4M3 byte: nearest, ties to even, satfinite (+-448), sign kept."""
    return _encode_nearest(v, E4M3_MAGNITUDES, 0x80)


def e8m0_ceil_exponent(s) -> np.ndarray:
    """Smallest integer e with 2^e >= s, for FP32 s > 0 (exact, via frexp:
    s = f * 2^x with f in [0.5, 1); s is a power of two iff f == 0.5)."""
    s = np.asarray(s, dtype=np.float32)
    f, x = np.frexp(s)
    return np.where(f == 0.5, x - 1, x).astype(np.int64)
