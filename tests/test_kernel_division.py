"""The encode kernel's two division shortcuts, checked on the CPU in exact
arithmetic: the block-scale quotient fl(b / 6) (rational arithmetic, below) and the
encode factor fl(S / sd) (integer arithmetic, at the end of this file).

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


def _rne_shift(N: np.ndarray, s: int) -> np.ndarray:
    """N / 2^s rounded to the nearest integer, ties to even (N >= 0)."""
    q = N >> s
    rem = N - (q << s)
    half = np.int64(1) << (s - 1)
    return q + ((rem > half) | ((rem == half) & ((q & 1) == 1)))


def _rne_to_24_bits(N: np.ndarray, sticky=None):
    """(M, s): N / 2^s rounded to 24 significant bits, ties to even, as M * 2^s with
    2^23 <= M <= 2^24 (sticky: a nonzero remainder below N's last bit)."""
    bl = np.floor(np.log2(N.astype(np.float64))).astype(np.int64) + 1
    bl = np.where((np.int64(1) << (bl - 1)) > N, bl - 1, bl)
    bl = np.where((np.int64(1) << bl) <= N, bl + 1, bl)
    s = bl - 24
    M = np.empty_like(N)
    for sv in np.unique(s):
        sel = s == sv
        n = N[sel]
        q = n >> sv
        rem = n - (q << sv)
        half = np.int64(1) << (sv - 1)
        st = np.zeros(n.shape, bool) if sticky is None else sticky[sel]
        M[sel] = q + ((rem > half) | ((rem == half) & (st | ((q & 1) == 1))))
    over = M == (1 << 24)
    return np.where(over, M >> 1, M), np.where(over, s + 1, s)


def test_scale_division_shortcut_equals_ieee_quotient_for_every_significand():
    """The encode factor e = fl(S / sd) for sd a positive E4M3 value: the kernel takes
    r = fl(1/sd), q0 = fl(S r), the residual S - q0 sd (one FMA, exact), and
    q1 = fl(q0 + residual r) (one FMA).  Checked here in exact integer arithmetic for
    every FP32 significand of S (2^23) against every E4M3 significand of sd that is not
    a power of two (1 + k/8, k = 1..7; a power of two makes r exact and the residual
    zero), with S in [1, 2).  Scaling S and sd by powers of two scales every step
    exactly while all intermediates stay normal, which the kernel ensures by taking
    this path only for S in [2^-90, 2^90] (sd lies in [2^-9, 448])."""
    Ms = np.arange(1 << 23, 1 << 24, dtype=np.int64)  # S = Ms / 2^23
    for md in range(9, 16):  # sd = md / 8
        num = 1 << 27  # r = RN(8 / md) in (0.5, 1): r = Mr / 2^24
        Mr, rr = divmod(num, md)
        if 2 * rr > md or (2 * rr == md and Mr % 2 == 1):
            Mr += 1
        P = Ms * Mr  # S r = P / 2^47, in (0.5, 2)
        ge1 = P >= (np.int64(1) << 47)
        Q = np.where(ge1, _rne_shift(P, 24), _rne_shift(P, 23))  # q0 = Q / 2^f
        f = np.where(ge1, 23, 24)
        R = (Ms << (f + 3 - 23)) - Q * md  # residual = R / 2^(f+3), exactly
        a = np.abs(R)
        while True:  # the residual fits in 24 significant bits (the FMA is exact)
            even = (a != 0) & ((a & 1) == 0)
            if not even.any():
                break
            a = np.where(even, a >> 1, a)
        assert (a < (1 << 24)).all()
        N = (Q << 27) + R * Mr  # q0 + residual r = N / 2^(f+27), exactly
        m1, s1 = _rne_to_24_bits(N)
        e1 = s1 - (f + 27)
        X = (Ms << 33) // md  # S / sd = (Ms 2^33 / md) / 2^53, with its remainder
        Xr = (Ms << 33) - X * md
        m2, s2 = _rne_to_24_bits(X, sticky=Xr > 0)
        e2 = s2 - 53
        bad = ~((m1 == m2) & (e1 == e2))
        assert not bad.any(), (md, int(bad.sum()), Ms[bad][:4])
