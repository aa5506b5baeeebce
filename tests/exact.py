"""Exact rational arithmetic helpers for pinning the oracle (test-only).

Values are Python ``Fraction``s; rounding to binary32 is done here from the
definition of the format (24-bit significand, exponents -126..127, gradual
underflow below 2^-126, overflow to infinity at 2^128 * (1 - 2^-25)), ties to
even.  Nothing here is shared with the oracle or with the CUDA library.
"""
from fractions import Fraction
import math

import numpy as np


def frac(x) -> Fraction:
    return Fraction(float(x))


def round_binary(q: Fraction, mant_bits: int, emin: int, emax: int):
    """Round rational q to a binary format with ``mant_bits`` significand bits
    (hidden bit included), nearest-even.  Returns a Fraction or +-inf float."""
    if q == 0:
        return Fraction(0)
    neg = q < 0
    a = -q if neg else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    E = max(e, emin)
    quantum = Fraction(2) ** (E - (mant_bits - 1))
    m = a / quantum
    r = m.numerator // m.denominator
    rem = m - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    v = r * quantum
    if v >= Fraction(2) ** (emax + 1):
        return -math.inf if neg else math.inf
    return -v if neg else v


def to_f32(q: Fraction) -> np.float32:
    v = round_binary(q, 24, -126, 127)
    return np.float32(float(v))


def exact_fma_f32(a, x, y) -> np.float32:
    """Correctly rounded binary32 a*x + y for finite inputs with a nonzero result."""
    q = frac(a) * frac(x) + frac(y)
    assert q != 0
    return to_f32(q)
