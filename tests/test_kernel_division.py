"""The encode kernel's shortcut for the block-scale quotient fl(b / 6), checked on
the CPU in exact rational arithmetic.

For BF16 inputs the block max b has at most 8 significant bits, and the kernel
replaces the IEEE division by q0 = fl(b * r) with r = fl(1/6), followed by one
FMA correction step q1 = fma(fma(-q0, 6, b), r, q0).  This test states that the
two agree for every positive finite BF16 value, subnormal quotients included, so
the kernel computes exactly the quotient that the recipe (and the oracle, which
divides) prescribes.  FP32 inputs keep the IEEE division in the kernel.
"""
from fractions import Fraction as Fr

import numpy as np


def rn32(x: Fr) -> Fr:
    """Round a rational to the nearest FP32 value, ties to even (subnormals too)."""
    if x == 0:
        return Fr(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    e = max(e, -126)
    ulp = Fr(2) ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    frac = q - n
    if frac > Fr(1, 2) or (frac == Fr(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_rn32_matches_numpy_float32():
    rng = np.random.default_rng(5)
    for v in rng.uniform(-1e3, 1e3, 200):
        f = Fr(float(v))
        assert float(rn32(f)) == float(np.float32(v))
    # a tie between two FP32 neighbours of 1 goes to the even one
    assert rn32(Fr(1) + Fr(1, 2 ** 24)) == 1
    assert rn32(Fr(1) + Fr(3, 2 ** 24)) == Fr(1) + Fr(2, 2 ** 23)


def test_reciprocal_constant_is_rounded_one_sixth():
    r = np.array([0x3E2AAAAB], np.uint32).view(np.float32)[0]
    assert Fr(float(r)) == rn32(Fr(1, 6))


def test_div6_short_equals_ieee_quotient_for_every_bf16():
    r = rn32(Fr(1, 6))
    bits = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    bad = []
    for v in bits:
        b = Fr(float(v))
        q0 = rn32(b * r)
        rem = rn32(b - q0 * 6)  # FMA: one rounding of the exact b - 6 q0
        assert rem == b - q0 * 6  # the residual is exact
        q1 = rn32(q0 + rem * r)
        if q1 != rn32(b / 6):
            bad.append(float(v))
    assert not bad, bad[:5]
