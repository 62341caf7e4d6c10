"""The block-scale arithmetic of the CUDA quantiser replaces the IEEE
division b / 6 (b = a block's largest magnitude, a bf16 value) by the
product with RN(1/6) and one fma residual correction.  This checks, in exact
rational arithmetic, that the corrected quotient is the correctly rounded
fp32 quotient for every non-negative finite bf16 b: +0, all subnormals and
all normals.  The rounding to fp32 is written out here (nearest, ties to
even, with the subnormal quantum 2^-149), so the check depends on no
floating-point unit."""
from fractions import Fraction

import numpy as np


def rn_f32(q: Fraction) -> Fraction:
    """q rounded to the nearest fp32 value, ties to even (no overflow)."""
    if q == 0:
        return Fraction(0)
    neg = q < 0
    a = -q if neg else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    return -r if neg else r


def bf16_value(bits: int) -> Fraction:
    exp = (bits >> 7) & 0xFF
    man = bits & 0x7F
    if exp == 0:
        return Fraction(man) * Fraction(2) ** (-133)
    return Fraction(128 + man) * Fraction(2) ** (exp - 134)


def test_rn_f32_against_numpy_on_samples():
    """The hand-written rounding agrees with numpy's fp32 conversion on
    values across the normal and subnormal ranges."""
    rng = np.random.default_rng(0)
    for v in np.concatenate([rng.normal(0, 1, 200), rng.normal(0, 1e-40, 200),
                             [1.0 / 3, 2.0 ** -149, 1.5 * 2.0 ** -149, 2.5 * 2.0 ** -149]]):
        assert float(rn_f32(Fraction(float(v)))) == float(np.float32(v)), v


def test_corrected_division_by_six_is_correctly_rounded_for_every_bf16():
    c = rn_f32(Fraction(1, 6))
    assert float(c) == float.fromhex("0x1.555556p-3")  # the kernel's constant
    for bits in range(0, 0x7F80):  # +0 .. the largest finite bf16
        b = bf16_value(bits)
        q0 = rn_f32(b * c)
        r = rn_f32(b - 6 * q0)
        q = rn_f32(r * c + q0)
        assert q == rn_f32(b / 6), hex(bits)
