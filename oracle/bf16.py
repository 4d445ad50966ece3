"""BF16 values in the oracle: decode, encode, round-to-nearest-even.

BF16 has 1 sign bit, an 8-bit exponent (bias 127, the binary32 range) and 7
stored significand bits, so 8 significant bits with the hidden bit.  Normal
values have exponents -126..127; subnormals are multiples of 2**-133.

PSI section II-C Eq.(5) states the rounding B as round-to-nearest,
ties-to-even; ``round_bf16`` rounds a float64 directly (no detour through
float32, which would round twice) and ``round_dyadic`` rounds an exact
rational n * 2**e, as in the exact evaluation of section IV-B Eq.(6).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

P = 8                 # significant bits, hidden bit included
EMIN = -126           # smallest normal exponent
QMIN = EMIN - (P - 1)  # -133: exponent of the subnormal spacing
EMAX = 127
OVERFLOW = 2.0 ** 128  # first magnitude that is not finite after rounding


def decode(bits) -> np.ndarray:
    """uint16 BF16 bit patterns -> float64 values (exact), from the fields."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    m = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + m / 128.0, (e - 127).astype(np.int32))
    sub = np.ldexp(m, QMIN)
    val = np.where(e == 0, sub, normal)
    val = np.where(e == 0xFF, np.where(m == 0, np.inf, np.nan), val)
    return sign * val


def encode(values) -> np.ndarray:
    """float64 values that are exactly BF16 -> uint16 bit patterns."""
    v = np.asarray(values, dtype=np.float64)
    f = v.astype(np.float32)  # exact for BF16-representable values
    if not np.array_equal(f.astype(np.float64), v, equal_nan=True):
        raise ValueError("encode: value is not representable in BF16")
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("encode: value is not representable in BF16")
    return (u >> 16).astype(np.uint16)


def round_bf16(x) -> np.ndarray:
    """B(x): float64 -> nearest BF16 (ties to even), returned as float64.

    The quantum of x is 2**(floor(log2|x|) - 7), floored at the subnormal
    spacing 2**-133.  Scaling by a power of two is exact, ``np.rint`` rounds
    half to even, and results of magnitude 2**128 or more overflow to inf.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                    # |x| = f * 2**e, 0.5 <= f < 1
    q = np.maximum(e - P, QMIN)           # floor(log2|x|) = e - 1
    r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    r = np.where(np.abs(r) >= OVERFLOW, np.copysign(np.inf, x), r)
    return np.where(np.isnan(x), np.nan, r)


def round_dyadic(n: int, e: int) -> float:
    """B(n * 2**e) for integers n, e, computed exactly with integers."""
    if n == 0:
        return 0.0
    sign = -1.0 if n < 0 else 1.0
    a = -n if n < 0 else n
    top = a.bit_length() - 1 + e          # floor(log2 |value|)
    q = max(top - (P - 1), QMIN)          # exponent of the last kept bit
    shift = q - e
    if shift <= 0:
        r = a << (-shift)
    else:
        r, rem = divmod(a, 1 << shift)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and (r & 1)):
            r += 1
    if r.bit_length() - 1 + q >= 128:
        return sign * math.inf
    return sign * math.ldexp(r, q)


def round_fraction(v: Fraction) -> float:
    """B(v) for a rational whose denominator is a power of two."""
    den = v.denominator
    if den & (den - 1):
        raise ValueError("round_fraction: denominator is not a power of two")
    return round_dyadic(v.numerator, -(den.bit_length() - 1))


def ulp(v) -> np.ndarray:
    """Spacing of BF16 values at magnitude |v| (2**-133 below the normal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    q = np.where(a == 0, QMIN, np.maximum(e - P, QMIN))
    return np.ldexp(1.0, q)
