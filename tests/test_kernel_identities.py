"""Arithmetic identities the step kernel relies on, checked exactly on the
CPU (rational arithmetic, no GPU): the variance code's dequantization q/255
without a table, as RN(q zh + RN(q zl)) with zh = RN(1/255) and
zl = RN(1/255 - zh), equals RN(q/255) for every code byte q."""

from fractions import Fraction

import numpy as np


def rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (normal
    range only, which is all these identities need)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert -126 <= e <= 127
    scale = Fraction(2) ** (e - 23)  # one unit in the last place
    n, r = divmod(a / scale, 1)
    n = int(n)
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * scale


def f32(x: float) -> Fraction:
    return Fraction(float(np.float32(x)))


def test_rn32_agrees_with_numpy_on_doubles():
    rng = np.random.default_rng(5)
    for x in rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000):
        assert rn32(Fraction(float(x))) == Fraction(float(np.float32(x)))


def test_variance_unit_value_without_a_table():
    zh = rn32(Fraction(1, 255))
    zl = rn32(Fraction(1, 255) - zh)
    # the kernel's constants, formed in double and rounded to fp32
    assert zh == f32(1.0 / 255.0)
    assert zl == f32(1.0 / 255.0 - float(np.float32(1.0 / 255.0)))
    for q in range(256):
        got = rn32(q * zh + rn32(q * zl)) if q else Fraction(0)
        assert got == (rn32(Fraction(q, 255)) if q else 0), q
