"""Buckets whose exact L2 norm sits at, just below or just above a binary32
rounding boundary (the midpoint between two adjacent binary32 values).

Construction: pick a midpoint m between binary32 neighbours f < f+, then
greedily write m^2 as a sum of binary32 squares (each element the largest
binary32 value whose square fits the remainder), so the exact sum of squares
ends a tiny remainder below m^2; one more small element pushes it just above
(or, where the remainder is itself a square, exactly onto m^2).  Used by the
oracle pins and by the GPU parity tests; built with exact rationals only.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from tests._exact import frac, sqrt_down_f32, sqrt_to_f32


def _bf16_down(x: np.float32) -> np.float32:
    """The bf16 value (as binary32) nearest to x towards zero."""
    return np.array([x], dtype=np.float32).view(np.uint32)[0] & np.uint32(0xFFFF0000)


def _to_f32_bits(b) -> np.float32:
    return np.array([b], dtype=np.uint32).view(np.float32)[0]


def midpoint_bucket(f: float, steps: int = 4, side: str = "below", bf16: bool = False):
    """Elements (binary32, or bf16 values held as binary32 with bf16=True) whose
    exact sum of squares lies within about 2^(-24 * steps) (2^(-8 * steps) for
    bf16) relative below the midpoint between f and its upper neighbour
    ('below'), just above it ('above'), and the value the norm must round to."""
    f = np.float32(f)
    fu = np.nextafter(f, np.float32(np.inf))
    m = (frac(f) + frac(fu)) / 2
    rem = m * m
    out = []
    for _ in range(steps):
        if rem <= Fraction(1, 2 ** 250):
            break
        x = sqrt_down_f32(rem)
        if bf16:
            x = _to_f32_bits(_bf16_down(x))
        if x == 0:
            break
        out.append(x)
        rem -= frac(x) * frac(x)
    if side == "above":
        # the smallest element whose square exceeds the remainder
        x = sqrt_to_f32(rem) if rem > 0 else np.float32(0)
        while frac(x) * frac(x) <= rem:
            x = np.nextafter(x, np.float32(np.inf))
        if bf16:
            b = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
            x = _to_f32_bits(((b + 0xFFFF) & 0xFFFF0000) if b & 0xFFFF else b)
        out.append(x)
    want = f if side == "below" else fu
    return np.array(out, dtype=np.float32), want


def exact_norm_f32(vals) -> np.float32:
    """binary32 rounding of the exact L2 norm of binary32 values."""
    s = sum((frac(v) * frac(v) for v in vals), Fraction(0))
    return sqrt_to_f32(s)
