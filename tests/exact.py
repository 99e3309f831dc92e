"""Exact rational helpers for the oracle pins (independent of oracle.formats)."""

from fractions import Fraction

import numpy as np


def exact_bf16_bits(v: Fraction) -> int:
    """Round an exact rational to BF16 (nearest, ties to even) with integer arithmetic."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2**e <= a < 2**(e+2)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 7)                            # 8 significant bits
    q = a / quantum
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * quantum
    f32 = np.float32(float(val))                                # exact: 8 significant bits
    assert Fraction(float(f32)) == val
    return sign | int(f32.view(np.uint32) >> 16)
