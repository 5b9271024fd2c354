"""Pins for the oracle's quantize / dequantize / grouped recipe (CPU only).

What pins what (none of these re-types the oracle's own formula):
  * hand-derived blocks in tests/golden/hand_blocks.json (closed-form cases);
  * amax            == numpy brute-force max|x| (exact, order free);
  * row-scaled with a constant per-row amax A == per-tensor with amax A
    ("NVFP4: enable row-scaled transpose quantization for backward", Greptile
    summary: the scalar case reproduces the earlier result bit for bit);
  * columnwise(X)   == rowwise(X^T) with the column amax (same PR, description:
    the columnwise output is the transposed quantization);
  * group-expanded amax == per-split per-tensor quantize, and zero-padded rows
    give zero codes / scales, ragged+padded == aligned ("Add NVFP4 four-over-six
    grouped GEMM for MoE training", description);
  * noop == 1 writes nothing ("row-scaled nvfp4 path: fuse row/col amax into a
    single TMA-tiled kernel", review comment and flowchart);
  * dequantize(quantize(x)) error within the FP4 half-step at the block scale,
    exact for on-grid inputs ("Add backward overrides and 1x16 weights to NVFP4
    four-over-six", description: dequantize formula);
  * four-over-six keeps the candidate with the smaller squared error, checked in
    float64 against the two single-candidate outputs;
  * 16x16 blocks: columnwise codes == transpose of rowwise codes, and 16x16 ==
    1x16 when every tile's 16 row maxima are equal.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.json")


def unpack(codes: np.ndarray, n: int) -> np.ndarray:
    """Packed bytes [lines][ceil(n/2)] -> nibbles [lines][n] (low nibble first)."""
    lo = codes & 0x0F
    hi = codes >> 4
    out = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    return out[:, :n]


def rng_matrix(rows, cols, seed, row_decades=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    if row_decades:
        x *= (10.0 ** rng.uniform(-row_decades, row_decades, (rows, 1))).astype(np.float32)
    return x


# ---------------------------------------------------------------- golden

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_derived_blocks(case):
    v = np.array(case["values"], np.float32)
    codes, scales = oracle.quantize_line(v, case["line_amax"], case["bound"],
                                         bool(case["four_over_six"]))
    assert list(scales) == case["scales"]
    assert list(codes) == case["codes"]
    if "dequant" in case:
        deq = oracle.dequantize(codes[None], scales[None], [case["line_amax"]], row_scaled=True,
                                rows=1, cols=len(v), bound=case["bound"])
        assert deq[0].tolist() == case["dequant"]


# ---------------------------------------------------------------- amax

@pytest.mark.parametrize("shape", [(1, 1), (3, 17), (33, 5), (64, 128), (0, 7), (7, 0)])
def test_amax_is_bruteforce_max(shape):
    x = rng_matrix(*shape, seed=1, row_decades=3)
    if x.size:
        x[0, 0] = -0.0
    r, c, t = oracle.amax(x)
    ax = np.abs(x.astype(np.float64))
    assert np.array_equal(r, ax.max(1) if shape[1] else np.zeros(shape[0]))
    assert np.array_equal(c, ax.max(0) if shape[0] else np.zeros(shape[1]))
    assert t == (ax.max() if x.size else 0.0)


def test_global_scale_closed_forms():
    assert oracle.global_scale(6.0, 448.0) == 448.0
    assert oracle.global_scale(6.0, 256.0) == 256.0
    assert oracle.global_scale(0.0, 448.0) == 1.0
    assert oracle.global_scale(1e-40, 448.0) == np.finfo(np.float32).max
    assert oracle.global_scale(2688.0, 448.0) == 1.0


def test_bf16_input_equals_widened_fp32_input():
    x = rng_matrix(40, 72, seed=2, row_decades=2)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    a = oracle.quantize(bits, "bf16")
    b = oracle.quantize(widened, "fp32")
    for d in ("row", "col"):
        for i in range(3):
            assert np.array_equal(a[d][i], b[d][i])


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("bound", [448.0, 256.0])
@pytest.mark.parametrize("fos", [False, True])
def test_constant_row_amax_row_scaled_equals_per_tensor(bound, fos):
    rows, cols, A = 48, 80, 3.25
    x = rng_matrix(rows, cols, seed=3)
    x = np.clip(x, -3.0, 3.0)
    x[np.arange(rows), np.arange(rows) % cols] = A * np.where(np.arange(rows) % 2, -1, 1)
    rs = oracle.quantize(x, mode=oracle.ROW_SCALED, bound=bound, four_over_six=fos,
                         columnwise=False)
    pt = oracle.quantize(x, mode=oracle.PER_TENSOR, bound=bound, four_over_six=fos,
                         columnwise=False)
    assert np.all(rs["row"][2] == A) and pt["row"][2][0] == A
    assert np.array_equal(rs["row"][0], pt["row"][0])
    assert np.array_equal(rs["row"][1], pt["row"][1])


@pytest.mark.parametrize("shape", [(37, 53), (64, 48), (16, 16), (1, 33), (33, 1)])
@pytest.mark.parametrize("mode", [oracle.ROW_SCALED, oracle.PER_TENSOR])
@pytest.mark.parametrize("fos", [False, True])
def test_columnwise_is_rowwise_of_transpose(shape, mode, fos):
    x = rng_matrix(*shape, seed=4, row_decades=2)
    col = oracle.quantize(x, mode=mode, four_over_six=fos, rowwise=False)["col"]
    xt = np.ascontiguousarray(x.T)
    _, ca, _ = oracle.amax(x)
    amax_in = ca if mode == oracle.ROW_SCALED else None
    row_t = oracle.quantize(xt, mode=mode, four_over_six=fos, columnwise=False,
                            row_amax_in=amax_in)["row"]
    for i in range(3):
        assert np.array_equal(col[i], row_t[i])


def test_line_max_gets_top_scale_and_code():
    # For every line, the block holding the line amax gets s8 = E4M3(448) (or
    # E4M3(256) with bound 256) and that element gets code +-6.
    x = rng_matrix(30, 70, seed=5, row_decades=4)
    for bound, top in ((448.0, 0x7E), (256.0, 0x78)):
        q = oracle.quantize(x, bound=bound, columnwise=False)["row"]
        nib = unpack(q[0], x.shape[1])
        for r in range(x.shape[0]):
            j = int(np.argmax(np.abs(x[r])))
            assert q[1][r, j // 16] == top
            assert nib[r, j] & 7 == 7 and (nib[r, j] >> 3) == (x[r, j] < 0)


def test_zero_rows_and_zero_tensor_quantize_to_zero():
    x = rng_matrix(64, 48, seed=6)
    x[::8] = 0.0
    q = oracle.quantize(x)
    assert np.all(q["row"][0][::8] == 0) and np.all(q["row"][1][::8] == 0)
    assert np.all(q["row"][2][::8] == 0)
    z = np.zeros((20, 36), np.float32)
    for mode in (oracle.ROW_SCALED, oracle.PER_TENSOR):
        q = oracle.quantize(z, mode=mode)
        for d in ("row", "col"):
            assert not q[d][0].any() and not q[d][1].any() and not q[d][2].any()


def test_noop_writes_nothing():
    x = rng_matrix(24, 40, seed=7)
    out = {"row": (np.full((24, 20), 0xA5, np.uint8), np.full((24, 3), 0xA5, np.uint8),
                   np.full(24, -1.0, np.float32)),
           "col": (np.full((40, 12), 0xA5, np.uint8), np.full((40, 2), 0xA5, np.uint8),
                   np.full(40, -1.0, np.float32))}
    oracle.quantize(x, noop=1.0, out=out)
    for d in ("row", "col"):
        assert np.all(out[d][0] == 0xA5) and np.all(out[d][1] == 0xA5)
        assert np.all(out[d][2] == -1.0)
    oracle.quantize(x, noop=0.0, out=out)
    assert not np.all(out["row"][2] == -1.0)


def test_tail_packing_odd_length():
    v = np.array([6.0] * 17, np.float32)
    codes, scales = oracle.quantize_line(v, 6.0)
    assert list(codes) == [0x77] * 8 + [0x07]
    assert list(scales) == [0x7E, 0x7E]


# ---------------------------------------------------------------- dequantize

def _block_bound(x, q_scales, amax_vec, bound, row_scaled):
    """Per element: half the E2M1 step at the block's encode scale, times the
    dequantize factor, with slack for FP32 rounding and for y above 6."""
    rows, cols = x.shape
    finv = np.float32(1.0) / np.float32(bound * 6.0)
    sd = oracle.e4m3_decode(q_scales).astype(np.float64)
    a = np.asarray(amax_vec, np.float64).reshape(-1)
    a = a[:, None] if row_scaled else a[0]
    D = sd * a * float(finv)                           # [rows][blocks]
    D = np.repeat(D, 16, axis=1)[:, :cols]
    return 1.0001 * D + 1e-30                          # half-step <= 1 code unit (y in [4,6])


@pytest.mark.parametrize("mode", [oracle.ROW_SCALED, oracle.PER_TENSOR])
@pytest.mark.parametrize("bound", [448.0, 256.0])
def test_dequantize_roundtrip_error_bound(mode, bound):
    x = rng_matrix(48, 100, seed=8, row_decades=2)
    q = oracle.quantize(x, mode=mode, bound=bound, columnwise=False)["row"]
    rs = mode == oracle.ROW_SCALED
    deq = oracle.dequantize(q[0], q[1], q[2], row_scaled=rs, rows=48, cols=100, bound=bound)
    err = np.abs(deq.astype(np.float64) - x)
    assert np.all(err <= _block_bound(x, q[1], q[2], bound, rs))
    # and the error is small relative to the block maximum: at most (1 + 2^-4) b / 6
    b = np.repeat(np.abs(np.pad(x, ((0, 0), (0, 12)))).reshape(48, -1, 16).max(2), 16, 1)[:, :100]
    assert np.all(err <= (1 + 2.0**-4) * b / 6 * 1.001 + 1e-30)


def test_dequantize_exact_for_grid_inputs():
    # values v * 2^k with v on the E2M1 grid and every block's max exactly 6 * 2^k,
    # so every block scale is 448 (or 256) and the encode factor is 2^-k
    rng = np.random.default_rng(9)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    x = rng.choice(grid, size=(16, 64)) * rng.choice([-1, 1], size=(16, 64))
    x[:, ::16] = 6.0
    x = (x * (2.0 ** rng.integers(-20, 20, size=(16, 1)))).astype(np.float32)
    for bound in (448.0, 256.0):
        q = oracle.quantize(x, bound=bound, columnwise=False)["row"]
        deq = oracle.dequantize(q[0], q[1], q[2], row_scaled=True, rows=16, cols=64, bound=bound)
        assert np.array_equal(deq, x)


def test_dequantize_bf16_is_rne_of_fp32():
    import torch
    x = rng_matrix(16, 48, seed=10, row_decades=3)
    q = oracle.quantize(x, columnwise=False)["row"]
    f = oracle.dequantize(q[0], q[1], q[2], row_scaled=True, rows=16, cols=48)
    h = oracle.dequantize(q[0], q[1], q[2], row_scaled=True, rows=16, cols=48, out_dtype="bf16")
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, want)


def test_dequantize_uses_scale_times_amax_first():
    # The dequantize formula of the torchao PR (description): (scale * amax) * factor_inv,
    # then the code value.  The two groupings differ for this scale/amax pair.
    f = np.float32
    finv = f(1) / f(2688)
    sd, a = f(oracle.e4m3_decode(np.array([0x31], np.uint8))[0]), f(0.7)
    first = f(f(sd * a) * finv)
    other = f(sd * f(a * finv))
    assert first != other
    codes = np.array([[0x07]], np.uint8)   # element 0: code 7 (6.0)
    deq = oracle.dequantize(codes, np.array([[0x31]], np.uint8), [a], row_scaled=True,
                            rows=1, cols=1)
    assert deq[0, 0] == f(f(6) * first)


# ---------------------------------------------------------------- four over six

def _sse64(x, codes, scales, amax_vec, bound, row_scaled):
    rows, cols = x.shape
    deq = oracle.dequantize(codes, scales, amax_vec, row_scaled=row_scaled, rows=rows, cols=cols,
                            bound=bound).astype(np.float64)
    d2 = (x.astype(np.float64) - deq) ** 2
    d2 = np.pad(d2, ((0, 0), (0, (-cols) % 16)))
    return d2.reshape(rows, -1, 16).sum(2)


@pytest.mark.parametrize("bound", [448.0, 256.0])
def test_four_over_six_keeps_lower_error_candidate(bound):
    x = rng_matrix(64, 160, seed=11, row_decades=2)
    lib = oracle.lib()
    rows, cols = x.shape
    outs = {}
    for fos in (0, 1, 2):
        codes = np.zeros((rows, (cols + 1) // 2), np.uint8)
        scales = np.zeros((rows, (cols + 15) // 16), np.uint8)
        r, _, _ = oracle.amax(x)
        for i in range(rows):
            lib.oracle_quantize_line(np.ascontiguousarray(x[i]), cols, 1, float(r[i]), bound,
                                     fos, codes[i], scales[i])
        outs[fos] = (codes, scales, r)
    e6 = _sse64(x, *outs[0], bound, True)
    e4 = _sse64(x, *outs[2], bound, True)
    ech = _sse64(x, *outs[1], bound, True)
    decided = np.abs(e4 - e6) > 1e-4 * np.maximum(e4, e6)
    want = np.where(e4 < e6, e4, e6)
    assert np.all(np.isclose(ech, want, rtol=1e-6, atol=0) | ~decided)
    assert np.all(ech <= np.maximum(e4, e6) * (1 + 1e-6))
    # both candidates are really exercised on this input
    chosen4 = np.isclose(ech, e4, rtol=1e-9) & decided & (e4 < e6)
    assert 0.05 < chosen4.mean() < 0.95
    # and with the option off the result is the T=6 candidate
    off = oracle.quantize(x, bound=bound, four_over_six=False, columnwise=False)["row"]
    assert np.array_equal(off[0], outs[0][0]) and np.array_equal(off[1], outs[0][1])


# ---------------------------------------------------------------- 16x16 blocks

@pytest.mark.parametrize("shape", [(64, 96), (40, 72), (17, 33)])
@pytest.mark.parametrize("fos", [False, True])
def test_2d_blocks_columnwise_is_transpose(shape, fos):
    x = rng_matrix(*shape, seed=12)
    q = oracle.quantize(x, mode=oracle.PER_TENSOR, block_2d=True, four_over_six=fos)
    rows, cols = shape
    rn = unpack(q["row"][0], cols)
    cn = unpack(q["col"][0], rows)
    assert np.array_equal(rn, cn.T)
    # one scale per 16x16 tile, replicated along the tile in both layouts
    rt = q["row"][1].reshape(rows, -1)
    ct = q["col"][1].reshape(cols, -1)
    for ti in range(-(-rows // 16)):
        for tj in range(-(-cols // 16)):
            s = rt[ti * 16:(ti + 1) * 16, tj]
            assert np.all(s == s[0]) and np.all(ct[tj * 16:(tj + 1) * 16, ti] == s[0])


def test_2d_blocks_reduce_to_1x16_when_row_maxima_equal():
    x = rng_matrix(64, 64, seed=13)
    x = np.clip(x, -2.5, 2.5)
    for ti in range(4):
        for tj in range(4):
            x[ti * 16:(ti + 1) * 16, tj * 16] = 2.5 + ti + tj   # same max in every row of the tile
    a = oracle.quantize(x, mode=oracle.PER_TENSOR, block_2d=True, columnwise=False)["row"]
    b = oracle.quantize(x, mode=oracle.PER_TENSOR, block_2d=False, columnwise=False)["row"]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_2d_blocks_reject_row_scaled():
    with pytest.raises(ValueError):
        oracle.quantize(rng_matrix(16, 16, 0), mode=oracle.ROW_SCALED, block_2d=True)


# ---------------------------------------------------------------- grouped

def _groups(rows_per_group, cols, seed, pad_to=None):
    rng = np.random.default_rng(seed)
    parts, ends, e = [], [], 0
    for n in rows_per_group:
        p = n if pad_to is None else -(-n // pad_to) * pad_to
        g = np.zeros((p, cols), np.float32)
        g[:n] = rng.standard_normal((n, cols)) * rng.uniform(0.01, 10)
        parts.append(g)
        e += p
        ends.append(e)
    return np.concatenate(parts), np.array(ends, np.int64)


@pytest.mark.parametrize("fos", [False, True])
def test_grouped_expanded_amax_equals_per_split_quantize(fos):
    x, ends = _groups([5, 0, 17, 3, 40], 48, seed=14)
    codes, scales, ra, ga = oracle.grouped_quantize_rowwise(x, "fp32", ends, bound=256.0,
                                                            four_over_six=fos)
    start = 0
    for g, end in enumerate(ends):
        if end > start:
            q = oracle.quantize(x[start:end], mode=oracle.PER_TENSOR, bound=256.0,
                                four_over_six=fos, columnwise=False)["row"]
            assert np.array_equal(codes[start:end], q[0])
            assert np.array_equal(scales[start:end], q[1])
            assert ga[g] == q[2][0]
            assert np.all(ra[start:end] == q[2][0])
        else:
            assert ga[g] == 0.0
        start = end


def test_grouped_ragged_padded_equals_aligned():
    counts = [7, 130, 0, 64, 1]
    xp, ends_p = _groups(counts, 64, seed=15, pad_to=128)
    q = oracle.grouped_quantize_rowwise(xp, "fp32", ends_p)
    # slice the real rows back out; quantize the unpadded ragged tensor
    keep = np.concatenate([np.arange(s, s + n) for s, n in
                           zip(np.concatenate([[0], ends_p[:-1]]), counts)])
    xr = xp[keep]
    ends_r = np.cumsum(counts).astype(np.int64)
    r = oracle.grouped_quantize_rowwise(xr, "fp32", ends_r)
    assert np.array_equal(q[0][keep], r[0]) and np.array_equal(q[1][keep], r[1])
    pad = np.setdiff1d(np.arange(xp.shape[0]), keep)
    assert not q[0][pad].any() and not q[1][pad].any()


def test_grouped_row_scaled_mode_equals_dense_row_scaled():
    x, ends = _groups([9, 23, 4], 40, seed=16)
    codes, scales, ra, _ = oracle.grouped_quantize_rowwise(x, "fp32", ends, mode=oracle.ROW_SCALED,
                                                           bound=448.0, four_over_six=False)
    d = oracle.quantize(x, mode=oracle.ROW_SCALED, columnwise=False)["row"]
    assert np.array_equal(codes, d[0]) and np.array_equal(scales, d[1])
    assert np.array_equal(ra, d[2])


@pytest.mark.parametrize("ends", [[5, 3, 36], [5, 20, 35], [-1, 36], [40]])
def test_grouped_rejects_bad_ends(ends):
    x = rng_matrix(36, 16, 0)
    with pytest.raises(ValueError):
        oracle.grouped_amax(x, "fp32", np.array(ends, np.int64))
