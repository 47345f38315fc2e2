"""Exact-arithmetic helpers for the pin tests: rationals and IEEE binary32 rounding.

These are written from the IEEE-754 definition of binary32 (24-bit significand,
exponent range [-126, 127], subnormals down to 2^-149, round to nearest, ties to
even); they share nothing with the oracle or with the CUDA library.
"""
from __future__ import annotations

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
