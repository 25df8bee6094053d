"""Exact rational rounding helpers used by tests to pin the oracle.

These are written from the IEEE 754 / OCP FP8 definitions of "round to the
nearest representable value, ties to the even significand" and work on
``fractions.Fraction`` values, so they are independent of both the C oracle
and the CUDA path.  Slow; for small inputs only.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def round_to_format(q: Fraction, precision: int, emin: int, max_finite: Fraction | None,
                    saturate: bool) -> Fraction:
    """Round ``q`` to the nearest value with ``precision`` significand bits
    (implicit bit included) and minimum normal exponent ``emin``; ties go to
    the even significand.  Beyond ``max_finite``: saturate, or return inf."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)                       # subnormals share the emin quantum
    quantum = Fraction(2) ** (e - (precision - 1))
    n = a / quantum
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * quantum
    if max_finite is not None and r > max_finite:
        if saturate:
            r = max_finite
        else:
            return Fraction(sign) * Fraction(10) ** 400  # stands for infinity
    return sign * r


F32_MAX = (2 - Fraction(1, 2 ** 23)) * Fraction(2) ** 127


def rn_f32(q: Fraction) -> Fraction:
    return round_to_format(q, 24, -126, F32_MAX, saturate=False)


def rn_bf16(q: Fraction) -> Fraction:
    return round_to_format(q, 8, -126, (2 - Fraction(1, 2 ** 7)) * Fraction(2) ** 127, saturate=False)


def rn_e4m3_sat(q: Fraction) -> Fraction:
    return round_to_format(q, 4, -6, Fraction(448), saturate=True)


def f32_of_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bits_of_f32(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def bf16_value(b: int) -> Fraction:
    return Fraction(f32_of_bits((b & 0xFFFF) << 16))
