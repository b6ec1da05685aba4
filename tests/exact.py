"""Exact rational arithmetic used to brute-force tiny cases in the tests.

Everything here follows the IEEE 754 and OCP FP8 definitions directly on
``fractions.Fraction`` values: no floating-point operation decides a result.
"""
from fractions import Fraction
import math
import struct


def frac(x: float) -> Fraction:
    return Fraction(float(x))


def round_half_even(q: Fraction) -> int:
    """Nearest integer to q, ties to even."""
    f = math.floor(q)
    rem = q - f
    if rem > Fraction(1, 2):
        return f + 1
    if rem < Fraction(1, 2):
        return f
    return f if f % 2 == 0 else f + 1


def to_f32(q: Fraction) -> float:
    """Round a rational to the nearest IEEE binary32, ties to even (no overflow handling:
    callers stay in range).  Returns the value as a Python float (exact)."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # correct the floating log estimate
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    k = round_half_even(a / quantum)
    return sign * float(k * quantum)


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def e4m3_magnitudes():
    """The 127 finite non-negative E4M3FN magnitudes, indexed by code 0x00..0x7E."""
    mags = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        if e == 0:
            mags.append(Fraction(m, 512))
        else:
            mags.append((1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return mags


_MAGS = e4m3_magnitudes()


def to_e4m3_code(q: Fraction, negative_zero: bool = False) -> int:
    """Nearest E4M3FN code to the rational q, ties to the even code, saturating
    at 448.  ``negative_zero`` gives the sign for q == 0."""
    neg = q < 0 or (q == 0 and negative_zero)
    a = abs(q)
    if a >= 448:
        return (0x80 if neg else 0) | 0x7E
    best = None
    for code, mag in enumerate(_MAGS):
        d = abs(mag - a)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return (0x80 if neg else 0) | best[1]


def e4m3_value(code: int) -> Fraction:
    mag = _MAGS[code & 0x7F]
    return -mag if code & 0x80 else mag


def round_format(q: Fraction, p: int, emin: int, emax: int):
    """Nearest value of a binary format with p significand bits, smallest normal
    exponent emin and largest exponent emax, ties to even, gradual underflow;
    beyond the largest finite value the result is +-inf (a float).  Returns a
    Fraction for finite results.  The sign of a zero result is not tracked."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, emin) - (p - 1))
    r = round_half_even(a / quantum) * quantum
    if r > (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax:
        return sign * math.inf
    return sign * r


BF16_FORMAT = (8, -126, 127)
FP16_FORMAT = (11, -14, 15)
