"""Pins for the oracle's GEMM consumer (CPU only).

The GEMM that consumes NVFP4 operands ("NVFP4: enable row-scaled transpose
quantization for backward", TransformerEngine PR #3206, sequence diagram: fprop
output times the activation's per-row amax and the weight's amax; wgrad output
times the outer product of both operands' per-line amax) is, by definition, the
matrix product of the two dequantized operands.  These tests tie oracle.gemm to
facts that do not come from its own code: hand-computed closed forms, identity
operands that must return the (separately pinned) dequantized other operand,
exact power-of-two scaling of one row or one column, linearity in K, and the
numpy product of the dequantize oracle's output.
"""
import numpy as np
import pytest

import oracle

F448 = 448.0 * 6.0  # 2688: amax == F makes amax / F exactly 1


def _op(codes, scales, amax, row_scaled=False, bound=448.0):
    return dict(codes=np.asarray(codes, np.uint8), scales=np.asarray(scales, np.uint8),
                amax=np.asarray(amax, np.float32).reshape(-1), row_scaled=row_scaled, bound=bound)


def _const(lines, k, code, scale, amax, bound=448.0):
    byte = (code & 15) | ((code & 15) << 4)
    return _op(np.full((lines, k // 2), byte), np.full((lines, k // 16), scale), [amax], False, bound)


def _identity(k, bound=448.0):
    """k x k operand whose values are exactly the identity matrix."""
    codes = np.zeros((k, k // 2), np.uint8)
    for i in range(k):
        codes[i, i // 2] |= (0x2 << 4) if i & 1 else 0x2  # E2M1 0x2 = 1.0
    return _op(codes, np.full((k, k // 16), 0x38), [bound * 6.0], False, bound)  # E4M3 0x38 = 1.0


def _random_operand(lines, k, seed, row_scaled, bound=448.0, four_over_six=False):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((lines, k)) * np.exp(rng.uniform(-3, 3, (lines, 1)))).astype(np.float32)
    mode = oracle.ROW_SCALED if row_scaled else oracle.PER_TENSOR
    o = oracle.quantize(x, "fp32", mode=mode, bound=bound, four_over_six=four_over_six,
                        columnwise=False)["row"]
    return _op(o[0], o[1], o[2], row_scaled, bound)


def test_constant_operands_closed_form():
    # every A value 6.0 (code 0x7, scale 1.0, amax/F = 1), every B value -1.0 (code 0xA)
    d = oracle.gemm(_const(3, 64, 0x7, 0x38, F448), _const(5, 64, 0xA, 0x38, F448))
    assert d.shape == (3, 5) and np.all(d == -384.0)  # 64 * 6 * -1
    # A value 0.5 * 2 (code 0x1, scale 0x40 = 2.0), B value 1.5 * 0.5 (code 0x3, scale 0x30 = 0.5),
    # B amax = 2F (factor 2) with bound 256: per product 1.0 * 1.5, K = 32
    d = oracle.gemm(_const(2, 32, 0x1, 0x40, F448),
                    _const(2, 32, 0x3, 0x30, 2 * 256.0 * 6.0, bound=256.0))
    assert np.all(d == 48.0)


def test_identity_b_returns_dequantized_a():
    a = _random_operand(6, 64, seed=1, row_scaled=True)
    d = oracle.gemm(a, _identity(64))
    deq = oracle.dequantize(a["codes"], a["scales"], a["amax"], row_scaled=True, rows=6, cols=64)
    # the dequantize oracle rounds to FP32 (and multiplies by fl(1/F)): a few ulp apart
    assert np.all(np.abs(d - deq) <= 2.0 ** -21 * np.abs(d))
    assert np.count_nonzero(d) > 300


def test_identity_a_returns_transposed_b():
    b = _random_operand(7, 32, seed=2, row_scaled=True, bound=256.0, four_over_six=True)
    d = oracle.gemm(_identity(32), b)
    deq = oracle.dequantize(b["codes"], b["scales"], b["amax"], row_scaled=True, rows=7, cols=32,
                            bound=256.0)
    assert d.shape == (32, 7)
    assert np.all(np.abs(d - deq.T) <= 2.0 ** -21 * np.abs(d))


def test_line_amax_scales_its_row_or_column_exactly():
    a = _random_operand(5, 48, seed=3, row_scaled=True)
    b = _random_operand(4, 48, seed=4, row_scaled=True)
    d = oracle.gemm(a, b)
    a2 = dict(a, amax=a["amax"].copy())
    a2["amax"][2] *= 2.0
    d2 = oracle.gemm(a2, b)
    assert np.array_equal(d2[2], 2.0 * d[2]) and np.array_equal(np.delete(d2, 2, 0), np.delete(d, 2, 0))
    b2 = dict(b, amax=b["amax"].copy())
    b2["amax"][1] *= 0.5
    d3 = oracle.gemm(a, b2)
    assert np.array_equal(d3[:, 1], 0.5 * d[:, 1])
    assert np.array_equal(np.delete(d3, 1, 1), np.delete(d, 1, 1))


def test_linear_in_k():
    a = _random_operand(3, 96, seed=5, row_scaled=True)
    b = _random_operand(4, 96, seed=6, row_scaled=False)
    d, dabs = oracle.gemm(a, b, with_abs=True)
    parts = []
    for lo, hi in ((0, 32), (32, 96)):
        ai = dict(a, codes=a["codes"][:, lo // 2:hi // 2], scales=a["scales"][:, lo // 16:hi // 16])
        bi = dict(b, codes=b["codes"][:, lo // 2:hi // 2], scales=b["scales"][:, lo // 16:hi // 16])
        parts.append(oracle.gemm(ai, bi))
    assert np.all(np.abs(parts[0] + parts[1] - d) <= 2.0 ** -48 * dabs)


def test_sign_bit_negates_a_row():
    a = _random_operand(3, 32, seed=7, row_scaled=True)
    b = _random_operand(2, 32, seed=8, row_scaled=True)
    d = oracle.gemm(a, b)
    a2 = dict(a, codes=a["codes"].copy())
    a2["codes"][1] ^= 0x88  # flip the sign bit of both nibbles
    assert np.array_equal(oracle.gemm(a2, b)[1], -d[1])


@pytest.mark.parametrize("row_scaled", [(True, True), (True, False), (False, True)])
def test_matches_product_of_dequantized_operands(row_scaled):
    a = _random_operand(9, 128, seed=9, row_scaled=row_scaled[0])
    b = _random_operand(11, 128, seed=10, row_scaled=row_scaled[1], bound=256.0, four_over_six=True)
    d, dabs = oracle.gemm(a, b, with_abs=True)
    da = oracle.dequantize(a["codes"], a["scales"], a["amax"], row_scaled=row_scaled[0], rows=9,
                           cols=128).astype(np.float64)
    db = oracle.dequantize(b["codes"], b["scales"], b["amax"], row_scaled=row_scaled[1], rows=11,
                           cols=128, bound=256.0).astype(np.float64)
    assert np.all(np.abs(da @ db.T - d) <= 2.0 ** -21 * dabs)
    assert np.all(dabs >= np.abs(d))


def test_grouped_gemm_is_the_per_group_product():
    """oracle.grouped_gemm against facts independent of its slicing: each group's rows
    equal the dense GEMM with its own expert (an empty group in between takes no
    rows and no expert rows); an expert's per-tensor amax scales exactly its group's
    rows; a single group is the dense GEMM."""
    k, n = 64, 8
    a = _random_operand(384, k, seed=21, row_scaled=True)
    experts = [_random_operand(n, k, seed=30 + g, row_scaled=False) for g in range(3)]
    b = _op(np.concatenate([e["codes"] for e in experts]),
            np.concatenate([e["scales"] for e in experts]),
            np.array([e["amax"][0] for e in experts], np.float32), False)
    ends = [128, 128, 384]  # group 1 empty
    d = oracle.grouped_gemm(a, b, ends, n)
    rows0 = dict(a, codes=a["codes"][:128], scales=a["scales"][:128], amax=a["amax"][:128])
    assert np.array_equal(d[:128], oracle.gemm(rows0, experts[0]))
    rows2 = dict(a, codes=a["codes"][128:], scales=a["scales"][128:], amax=a["amax"][128:])
    assert np.array_equal(d[128:], oracle.gemm(rows2, experts[2]))
    # doubling expert 2's amax doubles exactly rows 128..383
    b2 = dict(b, amax=b["amax"].copy())
    b2["amax"][2] *= 2.0
    d2 = oracle.grouped_gemm(a, b2, ends, n)
    assert np.array_equal(d2[128:], 2.0 * d[128:]) and np.array_equal(d2[:128], d[:128])
    # a single group is the dense GEMM with expert 0
    assert np.array_equal(oracle.grouped_gemm(a, b, [384], n), oracle.gemm(a, experts[0]))


def test_grouped_wgrad_sums_to_the_dense_product():
    """With one shared amax per line for every group (the same per-group values), the
    per-group K ranges add up to the dense GEMM over all of K (linearity in K), and an
    empty group's block is zero."""
    k = 96
    a = _random_operand(5, k, seed=41, row_scaled=True)
    b = _random_operand(6, k, seed=42, row_scaled=True)
    ends = [32, 32, 96]
    G = len(ends)
    ag = dict(a, amax=np.tile(a["amax"], G))
    bg = dict(b, amax=np.tile(b["amax"], G))
    d, dabs = oracle.grouped_gemm_wgrad(ag, bg, ends, with_abs=True)
    full, fabs = oracle.gemm(a, b, with_abs=True)
    assert np.all(d[1] == 0)
    assert np.all(np.abs(d.sum(0) - full) <= 2.0 ** -48 * fabs)
