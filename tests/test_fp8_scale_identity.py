"""The FP8 dispatch kernel computes the block scale amax / 448 without a
division: q0 = RN(amax * C) with C = RN(1/448), r = fma(-q0, 448, amax),
s = fma(r, C, q0). This file checks, for every non-negative finite bf16 value
of amax (amax is a bf16 value, so these are all the cases), that s is the
correctly rounded fp32 quotient RN(amax / 448) -- with exact rational
arithmetic emulating single-rounding fp32 FMA. CPU only."""
from __future__ import annotations

from fractions import Fraction

import numpy as np

C_BITS = 0x3B124925          # the constant the kernel uses


def rn32(v: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (no overflow here)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = Fraction(2) ** (max(e, -126) - 23)          # quantum (subnormal below 2^-126)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def f32(bits: int) -> Fraction:
    return Fraction(float(np.uint32(bits).view(np.float32)))


def test_constant_is_rn_of_one_over_448():
    assert f32(C_BITS) == rn32(Fraction(1, 448))


def test_scale_identity_all_bf16_amax():
    C = f32(C_BITS)
    bad = []
    for b16 in range(0, 0x7F80):                       # +0 .. largest finite bf16
        a = f32(b16 << 16)
        q0 = rn32(a * C)
        r = rn32(a - q0 * 448)                          # fma(-q0, 448, a)
        s = rn32(r * C + q0)                            # fma(r, C, q0)
        if s != rn32(a / 448):
            bad.append(b16)
    assert not bad, f"{len(bad)} bf16 amax values break the identity, e.g. {bad[:5]}"
