"""Exact rational arithmetic used to pin the oracle.

Nothing here calls the oracle or the CUDA library: values are computed with
``fractions.Fraction`` and rounded to binary32 by the IEEE 754 rule written
out with integers, so a wrong division, multiplication or rounding step on
either side shows up as a mismatch.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def rne_int(q: Fraction) -> int:
    """Round a rational to the nearest integer, ties to even."""
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def round_to_f32(a: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) binary32 value of ``a``,
    subnormals included; overflow gives +-inf."""
    if a == 0:
        return np.float32(0.0)
    sign = -1 if a < 0 else 1
    a = abs(a)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    if e < -126:
        q = rne_int(a * Fraction(2) ** 149)           # subnormal quantum 2^-149
        val = Fraction(q, 2 ** 149)
    else:
        q = rne_int(a * Fraction(2) ** (23 - e))      # 24-bit significand
        val = q * Fraction(2) ** (e - 23)
        if val >= Fraction(2) ** 128:
            return np.float32(sign * np.inf)
    # val is exactly representable in binary32, hence in binary64
    return np.float32(sign * float(val))


def f32(v) -> Fraction:
    """Exact rational value of a binary32 number."""
    return Fraction(float(np.float32(v)))


def quantize_row_exact(row_f32, mul=None, qmax=127):
    """Per-row symmetric quantization done with exact rationals plus one
    explicit binary32 rounding per operation of the definition:
    x' = fl(x*c), s = fl(amax/qmax), q = clamp(rne(fl(x'/s)), -qmax, qmax)
    (qmax = 127 for int8 codes, 7 for int4 ones)."""
    xs = [f32(v) for v in row_f32]
    if mul is not None:
        xs = [f32(round_to_f32(x * f32(c))) for x, c in zip(xs, mul)]
    amax = max(abs(x) for x in xs)
    s = round_to_f32(amax / qmax)
    if s == 0:
        return [0] * len(xs), np.float32(0.0)
    sF = f32(s)
    q = []
    for x in xs:
        v = rne_int(f32(round_to_f32(x / sF)))
        q.append(max(-qmax, min(qmax, v)))
    return q, s


def dequant_exact(acc: int, sx, sw) -> np.float32:
    """y = fl( fl(acc) * fl(sx*sw) ) with each rounding made explicit."""
    a = f32(round_to_f32(Fraction(int(acc))))
    sc = f32(round_to_f32(f32(sx) * f32(sw)))
    return round_to_f32(a * sc)
