"""Arithmetic identities the kernels rely on, proved over their whole input domain
in exact rational arithmetic (binary32 round-to-nearest-even, subnormals included).

The kernels replace a few correctly rounded operations of the spec by cheaper
sequences that give the same bits.  Each replacement is only valid because its
operand comes from a small set (a bf16 value), so the identity is checked
here for every member of that set.
"""
from fractions import Fraction

import numpy as np

R6 = Fraction(float(np.float32(1) / np.float32(6)))  # fl(1/6), the kernel's constant


def rn32(x: Fraction) -> Fraction:
    """Round an exact rational to the nearest binary32 value, ties to even (no overflow)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                       # below 2^-126 the spacing stays 2^-149
    q = a / Fraction(2) ** (e - 23)
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2):
        n += 1
    return sign * Fraction(n) * Fraction(2) ** (e - 23)


def test_block_amax_over_six_without_a_division():
    """t = fma(fma(-q0, 6, a), fl(1/6), q0) with q0 = fl(a * fl(1/6)) equals fl(a / 6)
    for every finite bf16 a >= 0 (the block amax is always such a value)."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    bad = []
    for v in vals.tolist():
        a = Fraction(v)
        q0 = rn32(a * R6)
        rem = rn32(a - 6 * q0)             # fma(-q0, 6, a)
        t = rn32(rem * R6 + q0)            # fma(rem, fl(1/6), q0)
        if t != rn32(a / 6):
            bad.append(v)
    assert not bad, f"{len(bad)} bf16 values break the identity, e.g. {bad[:5]}"
