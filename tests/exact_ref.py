"""Independent exact-arithmetic helpers for pinning the oracle (test-only).

Python integers and fractions, no numpy rounding: used to brute-force the
exact Hadamard sums on tiny inputs and to round them once to fp32.
"""
from fractions import Fraction

import numpy as np


def f32_to_fraction(v) -> Fraction:
    return Fraction(float(np.float32(v)))   # fp32 -> fp64 is exact


def round_fraction_to_f32(fr: Fraction) -> np.float32:
    """Nearest fp32 to an exact rational, ties to even (subnormals included)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    lsb = max(e - 23, -149)
    scaled = a / (Fraction(2) ** lsb)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    # n * 2^lsb is exactly representable in fp32 (n <= 2^24)
    return np.float32(sign * float(n) * 2.0 ** lsb)


def exact_signed_sum(h, v) -> np.float32:
    total = sum((int(hj) * f32_to_fraction(vj) for hj, vj in zip(h, v)),
                Fraction(0))
    return round_fraction_to_f32(total)
