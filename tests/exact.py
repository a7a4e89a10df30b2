"""Exact-arithmetic helpers for pinning the oracle (textbook definitions, independent of oracle/).

``round_f32`` rounds a rational to the nearest binary32 value, ties to even (IEEE 754 rounding to
a 24-bit significand, subnormals included).  ``f16_value`` decodes f16 bits through numpy.
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np

U32 = Fraction(1, 2 ** 24)          # unit roundoff of binary32


def f16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def f32_from_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def round_f32(v: Fraction) -> float:
    """Nearest binary32 to the rational v, ties to even (no overflow handling)."""
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp_exp = max(e, -126) - 23
    ulp = Fraction(2) ** ulp_exp
    q = a / ulp
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * ulp)


def gamma(m: int) -> float:
    u = 2.0 ** -24
    return m * u / (1 - m * u)
