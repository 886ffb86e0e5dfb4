"""Exact rational rounding to IEEE binary formats, for the oracle's pins.

A value is carried as a ``fractions.Fraction`` (exact), and ``round_binary``
returns the nearest value of a binary floating-point format with ``p``
significand bits and smallest normal exponent ``emin`` (ties to even,
subnormals on the fixed grid 2^(emin - p + 1), no overflow handling: callers
stay in range).  This is the IEEE-754 definition of a correctly rounded
operation, written with integers, so that a test can state what one binary32
(or binary16) operation must return without using the machine's float unit.
"""
from __future__ import annotations

from fractions import Fraction

F32 = (24, -126)
F16 = (11, -14)


def round_binary(x, fmt=F32) -> Fraction:
    p, emin = fmt
    x = Fraction(x)
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    step = Fraction(2) ** (max(e, emin) - (p - 1))
    q = a / step
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * step


def rf32(x) -> Fraction:
    """One binary32 rounding of an exact value."""
    return round_binary(x, F32)


def rf16(x) -> Fraction:
    """One binary16 rounding of an exact value."""
    return round_binary(x, F16)


def rint_even(x) -> int:
    """Nearest integer, ties to even (exact)."""
    x = Fraction(x)
    n = x.numerator // x.denominator           # floor
    rem = x - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def fr(v) -> Fraction:
    """Exact value of a numpy / Python float."""
    return Fraction(float(v))
