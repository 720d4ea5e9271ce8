"""The NVFP4 block scale needs RN32(amax / 6) for amax = max |y| of 16 BF16
values. The kernel forms it without an IEEE division: t = RN32(amax * c) with
c = RN32(1/6), the exact residual r = amax - 6 t from one FMA, then one
correction FMA q = RN32(t + r c) (Markstein's correction step for division by
a known divisor). This emulates those three operations in exact rational
arithmetic, rounding each result to FP32 by hand, and requires IEEE float32
division's result (numpy) for every non-negative finite BF16 value, subnormal
ones included."""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest FP32 value, ties to even (subnormals kept)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    assert Fraction(2) ** e <= x < Fraction(2) ** (e + 1)
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = x / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * ulp
    assert v < Fraction(2) ** 128
    return sign * v


def method(a: Fraction, c: Fraction) -> Fraction:
    t = rn32(a * c)
    r = rn32(a - 6 * t)          # fma(-t, 6, a)
    return rn32(t + r * c)       # fma(r, c, t)


def bf16_values() -> np.ndarray:
    bits = np.arange(0, 0x7F80, dtype=np.uint32)   # +0 .. largest finite, subnormals included
    return (bits << 16).view(np.float32)


def test_reciprocal_constant_is_rn32_of_one_sixth():
    c = np.float32(1.0) / np.float32(6.0)
    assert float(c) == float.fromhex("0x1.555556p-3")
    assert Fraction(float(c)) == rn32(Fraction(1, 6))


def test_three_operation_division_by_six_is_correctly_rounded_for_every_bf16():
    a32 = bf16_values()
    want = (a32 / np.float32(6.0)).astype(np.float32)   # IEEE division, correctly rounded
    c = Fraction(float.fromhex("0x1.555556p-3"))
    bad = []
    for a, w in zip(a32.tolist(), want.tolist()):
        q = method(Fraction(a), c)
        if q != Fraction(w):
            bad.append(a)
    assert not bad, f"{len(bad)} inputs differ, first {bad[:5]}"


def test_the_residual_is_exact():
    """r = amax - 6 t is representable, so one FMA gives it without rounding."""
    c = Fraction(float.fromhex("0x1.555556p-3"))
    for a in bf16_values()[::37].tolist():
        t = rn32(Fraction(a) * c)
        exact = Fraction(a) - 6 * t
        assert rn32(exact) == exact


def test_a_single_multiply_is_not_enough():
    """Without the correction step some quotients round the wrong way, so the
    test above would notice a dropped correction."""
    a32 = bf16_values()[0x3F80:0x4000]   # [1, 2)
    want = (a32 / np.float32(6.0)).astype(np.float32)
    got = (a32 * np.float32(float.fromhex("0x1.555556p-3"))).astype(np.float32)
    assert (got != want).any()
