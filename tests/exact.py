"""Exact-rational models of IEEE-754 rounding, for pinning the oracle.

Nothing here uses hardware floating-point arithmetic on the values being
checked: a binary32 or bfloat16 result is found by rounding an exact rational
(Python ``Fraction``) to the nearest representable value, ties to even, from
the formats' definitions (binary32: 24-bit significand, exponents -126..127;
bfloat16: 8-bit significand, same exponent range).
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bits_f32(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def exact(x) -> Fraction:
    """Exact value of a finite float32 / Python float."""
    return Fraction(float(x))


def _round_to_format(r: Fraction, sig_bits: int, emin: int = -126, emax: int = 127):
    """Magnitude of the nearest value to |r| with a sig_bits-bit significand
    (including the leading bit), subnormals below 2**emin, inf beyond the
    largest finite value. Returns a non-negative Fraction or float('inf')."""
    a = abs(r)
    if a == 0:
        return Fraction(0)
    # exponent e with 2**e <= a < 2**(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (sig_bits - 1))
    m = a / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    largest = (2 - Fraction(2) ** (1 - sig_bits)) * Fraction(2) ** emax
    if v > largest:
        return float("inf")
    return v


def _signed_f32(mag, negative: bool) -> np.float32:
    v = np.float32(float(mag))
    return np.float32(-v) if negative else v


def rn_f32(r: Fraction, negative_zero: bool = False) -> np.float32:
    """Nearest binary32 to r; an exact zero takes the sign given."""
    if r == 0:
        return _signed_f32(0, negative_zero)
    return _signed_f32(_round_to_format(r, 24), r < 0)


def rn_bf16_bits(x) -> int:
    """bfloat16 bit pattern of the nearest bfloat16 to the float32 value x
    (ties to even; the sign of zero is kept)."""
    x = np.float32(x)
    negative = bool(np.signbit(x))
    if x == 0:
        mag = Fraction(0)
    else:
        mag = _round_to_format(exact(x), 8)
    if mag == float("inf"):
        bits = 0x7F80
    else:
        b = f32_bits(np.float32(float(mag)))
        assert b & 0xFFFF == 0, "a bfloat16 value has a zero lower half"
        bits = b >> 16
    return bits | (0x8000 if negative else 0)


def rn_f16_bits(x) -> int:
    """IEEE binary16 bit pattern of the nearest binary16 to the float32 value
    x (ties to even; 11-bit significand, exponents -14..15, subnormals down to
    2**-24; beyond the largest finite value, inf; the sign of zero is kept)."""
    x = np.float32(x)
    negative = bool(np.signbit(x))
    mag = Fraction(0) if x == 0 else _round_to_format(exact(x), 11, emin=-14, emax=15)
    if mag == float("inf"):
        bits = 0x7C00
    elif mag == 0:
        bits = 0
    else:
        e = mag.numerator.bit_length() - mag.denominator.bit_length()
        if Fraction(2) ** e > mag:
            e -= 1
        if e < -14:                       # subnormal: fraction * 2**-24
            frac = mag / Fraction(2) ** -24
            assert frac.denominator == 1
            bits = int(frac)
        else:
            m = mag / Fraction(2) ** (e - 10)
            assert m.denominator == 1 and 1024 <= m < 2048
            bits = ((e + 15) << 10) | (int(m) - 1024)
    return bits | (0x8000 if negative else 0)


def f16_value(bits: int) -> Fraction | float:
    """Exact value of a finite binary16 bit pattern (inf for infinities)."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    if e == 0x1F:
        return sign * float("inf")
    if e == 0:
        return sign * Fraction(f) * Fraction(2) ** -24
    return sign * Fraction(f + 1024) * Fraction(2) ** (e - 25)


def _neg(x) -> bool:
    return bool(np.signbit(np.float32(x)))


def mul_model(a, b) -> np.float32:
    """IEEE binary32 product of two finite binary32 values, from exact arithmetic."""
    r = exact(a) * exact(b)
    return rn_f32(r, negative_zero=_neg(a) != _neg(b))


def add_model(a, b) -> np.float32:
    """IEEE binary32 sum (round to nearest) of two finite binary32 values."""
    r = exact(a) + exact(b)
    # an exact zero sum is -0 only when both addends are -0
    return rn_f32(r, negative_zero=(_neg(a) and _neg(b) and a == 0 and b == 0))


def sub_model(a, b) -> np.float32:
    return add_model(a, -np.float32(b))


def rotate_pair_model(e, o, c, s):
    """Eager-order pair rotation from exact products and sums, each rounded
    once to binary32: y0 = RN(RN(e*c) - RN(o*s)), y1 = RN(RN(e*s) + RN(o*c))."""
    e, o, c, s = (np.float32(v) for v in (e, o, c, s))
    p1 = mul_model(e, c)
    p2 = mul_model(o, s)
    p3 = mul_model(e, s)
    p4 = mul_model(o, c)
    return sub_model(p1, p2), add_model(p3, p4)
