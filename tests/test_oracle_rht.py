"""Pins for the oracle's random Hadamard transform of the columnwise operand (CPU).

TE-3206's description names the transform, as something that PR leaves out of the
transposed path, but does not define it; the oracle's reading R14 is
y = (1/4) H16 diag(s) x per column and per block of 16 rows, H16 the Sylvester
Hadamard matrix, in FP32 butterfly steps.  These
tests tie oracle.rht16 to facts outside its code: scipy's Hadamard matrix on inputs
whose products and sums are exact in FP32, the FP64 product within the butterfly's
rounding bound, orthonormality (the transform applied twice is the identity; the
product of two transformed operands is the product of the originals), the image of
a single spike, the sign mask, and block locality.
"""
import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle

H16 = hadamard(16).astype(np.float64)


def _signs(mask):
    return np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])


def _reference(x, mask):
    """FP64: (1/4) H16 diag(s) applied to each 16-row block of each column."""
    rows, cols = x.shape
    m = 0.25 * H16 @ np.diag(_signs(mask))
    return np.concatenate([m @ x[r:r + 16].astype(np.float64) for r in range(0, rows, 16)])


@pytest.mark.parametrize("mask", [0x0000, 0xFFFF, 0x8421, 0x1234, 0xBEEF])
def test_matches_scipy_hadamard_exactly_on_integers(mask):
    rng = np.random.default_rng(mask)
    x = rng.integers(-1024, 1025, size=(64, 7)).astype(np.float32)  # sums stay exact in FP32
    assert np.array_equal(oracle.rht16(x, "fp32", mask).astype(np.float64), _reference(x, mask))


def test_within_the_butterfly_rounding_bound():
    """Four levels of FP32 additions: each output is within 4 u sum|x| / 4 of the
    exact value (u = 2^-24), plus nothing for the exact product with 1/4."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((256, 33)) * np.exp(rng.uniform(-6, 6, (256, 1)))).astype(np.float32)
    y = oracle.rht16(x, "fp32", 0x5A5A).astype(np.float64)
    ref = _reference(x, 0x5A5A)
    absx = np.abs(x.astype(np.float64))
    mag = np.concatenate([np.repeat(absx[r:r + 16].sum(0, keepdims=True), 16, 0)
                          for r in range(0, 256, 16)])
    assert np.all(np.abs(y - ref) <= 4 * 2.0 ** -24 * 0.25 * mag)
    assert np.count_nonzero(y != ref) > 0  # the bound is not vacuous: rounding happens


def test_applied_twice_is_the_identity_without_signs():
    rng = np.random.default_rng(2)
    x = rng.integers(-512, 513, size=(48, 5)).astype(np.float32)
    y = oracle.rht16(oracle.rht16(x, "fp32", 0), "fp32", 0)
    assert np.array_equal(y, x)  # (H/4)(H/4) = I, exact on these integers


def test_a_spike_spreads_to_a_signed_hadamard_column():
    x = np.zeros((32, 3), np.float32)
    x[16 + 5, 1] = 64.0
    mask = 0x0020  # flips row 5 of each block
    y = oracle.rht16(x, "fp32", mask)
    assert np.all(y[:16] == 0) and np.all(y[:, [0, 2]] == 0)
    assert np.array_equal(y[16:, 1], (-0.25 * 64.0 * H16[:, 5]).astype(np.float32))
    assert np.all(np.abs(y[16:, 1]) == 16.0)  # the spike's magnitude divided by 4, everywhere


def test_full_sign_mask_negates_the_output():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 9)).astype(np.float32)
    assert np.array_equal(oracle.rht16(x, "fp32", 0xFFFF), -oracle.rht16(x, "fp32", 0))


def test_blocks_and_columns_are_independent():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 6)).astype(np.float32)
    y = oracle.rht16(x, "fp32", 0x0F0F)
    x2 = x.copy()
    x2[40, 3] += 1.0  # block 2 of column 3
    y2 = oracle.rht16(x2, "fp32", 0x0F0F)
    changed = np.argwhere(y2 != y)
    assert changed.size and set(map(tuple, changed[:, ::-1] // [1, 16])) == {(3, 2)}


def test_product_of_transformed_operands_is_the_original_product():
    """The wgrad identity the transform relies on: with the same signs on both
    operands, (Q dY)^T (Q X) = dY^T X because Q is orthonormal."""
    rng = np.random.default_rng(5)
    dy = rng.standard_normal((128, 6)).astype(np.float32)
    x = rng.standard_normal((128, 4)).astype(np.float32)
    a = oracle.rht16(dy, "fp32", 0x3C5A).astype(np.float64)
    b = oracle.rht16(x, "fp32", 0x3C5A).astype(np.float64)
    exact = dy.astype(np.float64).T @ x.astype(np.float64)
    mag = np.abs(dy.astype(np.float64)).T @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(a.T @ b - exact) <= 2.0 ** -19 * mag)


def test_bf16_input_is_widened_first():
    rng = np.random.default_rng(6)
    f = rng.standard_normal((32, 4)).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(oracle.rht16(bits, "bf16", 0x77), oracle.rht16(widened, "fp32", 0x77))


def test_rows_not_a_multiple_of_16_are_rejected():
    with pytest.raises(ValueError):
        oracle.rht16(np.zeros((24, 4), np.float32))


def test_columnwise_quantize_of_the_transform():
    """quantize_columnwise_rht is the columnwise quantization of the transformed
    operand: its per-column amax is the exact max |y| of the transformed column."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 5)) * 0.1).astype(np.float32)
    x[3, 2] = 50.0  # an outlier the transform spreads over its block
    codes, scales, amax = oracle.quantize_columnwise_rht(x, "fp32", 0x1111)
    y = oracle.rht16(x, "fp32", 0x1111)
    assert np.array_equal(amax, np.abs(y).max(0))
    assert amax[2] < 50.0 / 4 + 1.0  # the outlier's block amax is about a quarter of it
    ref = oracle.quantize(y, "fp32", rowwise=False)["col"]
    assert np.array_equal(codes, ref[0]) and np.array_equal(scales, ref[1])
