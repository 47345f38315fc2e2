"""Exact-arithmetic helpers for the pin tests: rationals and IEEE binary32 rounding.

These are written from the IEEE-754 definition of binary32 (24-bit significand,
exponent range [-126, 127], subnormals down to 2^-149, round to nearest, ties to
even); they share nothing with the oracle or with the CUDA library.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def frac(x) -> Fraction:
    """Exact rational value of a finite float32 / float64."""
    return Fraction(float(x))


def round_half_even(fr: Fraction) -> int:
    """Nearest integer to a rational, ties to even."""
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def to_f32(fr: Fraction) -> np.float32:
    """Round a rational to the nearest binary32 value, ties to even (no overflow)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                    # subnormal range shares the 2^-126 binade quantum
    quantum = Fraction(2) ** (e - 23)
    m = round_half_even(a / quantum)
    val = m * quantum
    return np.float32(sign * float(val))


def ulp32(x) -> float:
    """Spacing of float32 numbers at |x| (at least the smallest subnormal)."""
    return float(np.spacing(np.float32(abs(float(x)))))


def dist_to_half_integer(fr: Fraction) -> Fraction:
    fl = fr.numerator // fr.denominator
    return abs(fr - fl - Fraction(1, 2))


def sqrt_to_f32(s: Fraction) -> np.float32:
    """The binary32 value nearest (ties to even) to the square root of a
    nonnegative rational whose denominator is a power of two no larger than
    2^600: the integer square root of s * 2^600 brackets the root within
    2^-300, far below half the smallest binary32 quantum (2^-150), so the
    rounding of the bracket's midpoint equals the rounding of the root unless
    the root is exact, which the remainder tells."""
    j = 300
    x = s * Fraction(4) ** j
    assert x.denominator == 1 and x >= 0
    r = math.isqrt(x.numerator)
    if r * r == x.numerator:
        return to_f32(Fraction(r, 2 ** j))
    return to_f32(Fraction(2 * r + 1, 2 ** (j + 1)))


def sqrt_down_f32(s: Fraction) -> np.float32:
    """The largest binary32 value whose square does not exceed s (s >= 0)."""
    x = sqrt_to_f32(s)
    while frac(x) * frac(x) > s:
        x = np.nextafter(x, np.float32(0))
    return np.float32(x)
