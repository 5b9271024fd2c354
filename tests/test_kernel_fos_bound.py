"""The encode kernel's bounded four-over-six decision, checked on the CPU.

Four-over-six keeps the block's T = 4 candidate when its squared error is below the
T = 6 one ("Add NVFP4 four-over-six grouped GEMM for MoE training", torchao PR #9,
description), each error being the FP32 sum, in element order, of
fl(x_i - fl(v_i D))^2 with D the block's dequantize factor ("Add backward overrides
and 1x16 weights to NVFP4 four-over-six", torchao PR #8, description).  The kernel
first compares estimates E' = fl(fl(D D) A), A the sum of the squared residuals of
the scaled values, r_i = fl(v_i - y_i) with y_i = fl(x_i e), accumulated as two
8-term FMA chains (even and odd i) and their sum.  Its proof bounds |err - E'| by
2096.4 u D^2 (u = 2^-24) when fl(b e) <= 6.5 for both candidates and D lies in
[2^-62, 2^61]; it then keeps T = 4 when E'4 - E'6 < -2^-12 (D4^2 + D6^2), keeps
T = 6 when the difference exceeds +2^-12 (D4^2 + D6^2), and sums exactly otherwise.

This test restates that arithmetic with NumPy FP32 operations (the FMA as an exact
FP64 product plus the addend, rounded to FP32: a double rounding that can differ
from the hardware's by one unit in the last place, far inside the bound) and checks,
over blocks of several shapes, that the estimate stays inside the proven bound,
that a decision the bound makes never contradicts the exact comparison, and that
the bound leaves few ordinary blocks to the exact sums.
"""
import zlib

import numpy as np
import pytest

import oracle

f32 = np.float32
U = 2.0 ** -24
PROVEN = 2096.4  # |err - E'| <= PROVEN * u * D^2 inside the guarded range
TOL = 2.0 ** -12


def candidate_errors(x: np.ndarray, a: np.ndarray, bound: float):
    """Per block of x [n, 16] (FP32) with line amax a [n]: for T = 6 and T = 4 the
    exact error, the estimate E', D, and fl(b e); and the scale bytes."""
    n = x.shape[0]
    F = f32(bound * 6.0)
    F_inv = f32(1.0) / F
    S = (F / a).astype(f32)
    b = np.abs(x).max(axis=1).astype(f32)
    out = {}
    for T in (6, 4):
        s32 = ((b / f32(T)).astype(f32) * S).astype(f32)
        s8 = oracle.e4m3_encode(s32)
        sd = oracle.e4m3_decode(s8).astype(f32)
        e = np.where(sd == 0, f32(0), S / np.where(sd == 0, f32(1), sd)).astype(f32)
        y = (x * e[:, None]).astype(f32)
        v = oracle.e2m1_decode(oracle.e2m1_encode(y.ravel())).reshape(y.shape).astype(f32)
        D = ((sd * a).astype(f32) * F_inv).astype(f32)
        d = (x - (v * D[:, None]).astype(f32)).astype(f32)
        p = (d * d).astype(f32)
        err = np.zeros(n, f32)
        for i in range(16):
            err = (err + p[:, i]).astype(f32)
        r = (v - y).astype(f32)
        acc = [np.zeros(n, f32), np.zeros(n, f32)]
        for i in range(16):
            ri = r[:, i].astype(np.float64)
            acc[i & 1] = (ri * ri + acc[i & 1].astype(np.float64)).astype(f32)
        A = (acc[0] + acc[1]).astype(f32)
        est = ((D * D).astype(f32) * A).astype(f32)
        out[T] = dict(err=err, est=est, D=D, ymax=(b * e).astype(f32), s8=s8)
    return out


def decide(c):
    """The kernel's decision: 1 (T = 4), 0 (T = 6) or -1 (exact sums).  The kernel
    checks fl(b e6) <= 6.5, D6 >= 2^-62 and D4 <= 2^61 only: the T = 4 scale is never
    below the T = 6 one, so the same bounds then hold for the other candidate (checked
    here on every block)."""
    c6, c4 = c[6], c[4]
    full = (c6["ymax"] <= 6.5) & (c4["ymax"] <= 6.5)
    for D in (c6["D"], c4["D"]):
        full &= (D >= 2.0 ** -62) & (D <= 2.0 ** 61)
    ok = (c6["ymax"] <= 6.5) & (c6["D"] >= 2.0 ** -62) & (c4["D"] <= 2.0 ** 61)
    assert np.array_equal(ok, full)
    q6 = (c6["D"] * c6["D"]).astype(f32)
    q4 = (c4["D"] * c4["D"]).astype(f32)
    diff = (c4["est"] - c6["est"]).astype(f32)
    with np.errstate(invalid="ignore", over="ignore"):
        tol = (f32(TOL) * (q4 + q6).astype(f32)).astype(f32)
        pick = np.where(diff < -tol, 1, np.where(diff > tol, 0, -1))
    pick = np.where(ok, pick, -1)
    return np.where(c6["s8"] == c4["s8"], 0, pick), ok


def blocks(kind, n, rng):
    if kind == "normal":
        x = rng.standard_normal((n, 16))
    elif kind == "heavy":
        x = rng.standard_normal((n, 16))
        x[rng.random((n, 16)) < 0.02] *= 30
    elif kind == "uniform":
        x = rng.uniform(-1, 1, (n, 16))
    elif kind == "halves":
        x = rng.integers(-12, 13, (n, 16)) * 0.5
    else:  # wide dynamic range inside a block
        x = rng.standard_normal((n, 16)) * np.exp(rng.uniform(-12, 12, (n, 16)))
    return x.astype(f32)


@pytest.mark.parametrize("kind", ["normal", "heavy", "uniform", "halves", "wide"])
@pytest.mark.parametrize("bound", [256.0, 448.0])
@pytest.mark.parametrize("bf16", [False, True])
def test_bounded_decision_agrees_with_exact_sums(kind, bound, bf16):
    rng = np.random.default_rng(zlib.crc32(f"{kind}/{bound}/{bf16}".encode()))
    x = blocks(kind, 40_000, rng)
    if bf16:
        x = oracle.bf16_to_f32(oracle.f32_to_bf16(x)).astype(f32)
    b = np.abs(x).max(axis=1)
    a = np.where(b > 0, b * rng.uniform(1.0, 30.0, len(b)), 1.0).astype(f32)
    c = candidate_errors(x, a, bound)
    pick, ok = decide(c)
    for T in (6, 4):
        gap = np.abs(c[T]["err"].astype(np.float64) - c[T]["est"]) / c[T]["D"].astype(np.float64) ** 2
        assert gap[ok].max(initial=0.0) <= PROVEN * U
    four = c[4]["err"] < c[6]["err"]
    assert not np.any((pick == 1) & ~four)
    assert not np.any((pick == 0) & four)
    if kind in ("normal", "heavy", "uniform"):
        assert (pick < 0).mean() < 0.02  # ordinary blocks: the bound nearly always decides


def test_guard_sends_saturated_and_tiny_blocks_to_exact_sums():
    """A given amax below the block max saturates the codes (|y| > 6.5), and a
    dequantize factor below 2^-62 is outside the analysed range: both go exact."""
    rng = np.random.default_rng(3)
    x = blocks("normal", 1000, rng)
    b = np.abs(x).max(axis=1)
    c = candidate_errors(x, (b * 0.25).astype(f32), 256.0)
    _, ok = decide(c)
    assert not ok.any()
    xt = (x * f32(2.0 ** -70)).astype(f32)
    bt = np.abs(xt).max(axis=1)
    c = candidate_errors(xt, bt.astype(f32), 256.0)
    _, ok = decide(c)
    assert not ok.any()
