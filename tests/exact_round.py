"""Exact rational rounding used by the pins of the element encode: the FP32
quotient x / t rounded once, from the definition of the format, and the E2M1 code
of it by brute force over the eight magnitudes.  Test infrastructure; it shares
nothing with the oracle or the CUDA library."""
import math
from fractions import Fraction

import numpy as np

E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def rn32(q: Fraction) -> float:
    """The FP32 value nearest to the rational q (ties to the even significand):
    24-bit significands, exponents down to -126 with the subnormal grid 2^-149
    below, infinity past the largest finite value."""
    if q == 0:
        return 0.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    n = a / ulp
    k = n.numerator // n.denominator
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    v = k * ulp
    if v > Fraction(float(np.finfo(np.float32).max)):
        return math.copysign(math.inf, q)
    return math.copysign(float(v), q)


def e2m1_nearest(v: float) -> int:
    """Brute force: the E2M1 code whose value is nearest v (ties to the even
    magnitude index), saturating at 6; the sign bit is the sign bit of v."""
    sign = 8 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    best = min(range(8), key=lambda i: (abs(E2M1_MAGS[i] - a), i % 2, i))
    return sign | best


def code_of_quotient(x, t) -> int:
    """e2m1(RN(x / t)); a zero t gives the signed zero of x."""
    x, t = float(np.float32(x)), float(np.float32(t))
    if t == 0:
        return 8 if math.copysign(1.0, x) < 0 else 0
    q = rn32(Fraction(x) / Fraction(t))
    if q == 0:
        return 8 if math.copysign(1.0, x) < 0 else 0
    return e2m1_nearest(q)
