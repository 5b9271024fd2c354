"""Seeded random sweep of the quantize calls against the oracle (GPU, through the C
ABI), byte for byte: shapes drawn around the tile edges (multiples of 16, 32, 64
and 128, plus or minus one) and anywhere, both input types, both modes, each
direction alone and both, four-over-six with either bound, 16x16 blocks, inputs that
start at an odd element (the plain-load paths), and the transform's calls.  Every
case is drawn from one seed, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads
from gpu_helpers import assert_same, cfg, gpu_quantize, host_bits, oracle_quantize

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dim(rng, hi):
    """A size near a tile edge (often) or anywhere below hi."""
    if rng.random() < 0.6:
        base = int(rng.choice([16, 32, 64, 128, 256, 384, 512]))
        return max(1, min(hi, base + int(rng.choice([-1, 0, 0, 1]))))
    return int(rng.integers(1, hi + 1))


def _case(i):
    rng = np.random.default_rng(1000 + i)
    rows, cols = _dim(rng, 700), _dim(rng, 900)
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    mode = nv.NVFP4_ROW_SCALED if rng.random() < 0.6 else nv.NVFP4_PER_TENSOR
    fos = bool(rng.random() < 0.4)
    bound = 256.0 if (fos and rng.random() < 0.5) else 448.0
    b2d = bool(mode == nv.NVFP4_PER_TENSOR and rng.random() < 0.3)
    direction = str(rng.choice(["both", "both", "row", "col"]))
    offset = int(rng.random() < 0.2)  # start one element into a wider buffer
    decades = float(rng.choice([0.0, 1.0, 3.0]))
    return rows, cols, dtype, mode, fos, bound, b2d, direction, offset, decades


@pytest.mark.parametrize("i", range(80))
def test_random_quantize_matches_oracle(i):
    rows, cols, dtype, mode, fos, bound, b2d, direction, offset, decades = _case(i)
    x = workloads.seeded_normal(rows, cols, seed=2000 + i, dtype=dtype, device=DEV,
                                row_scale_decades=decades)
    if offset:  # the same matrix, contiguous, one element into a buffer
        buf = torch.empty(rows * cols + 1, dtype=dtype, device=DEV)
        buf[1:].copy_(x.reshape(-1))
        x = buf[1:].view(rows, cols)
    c = cfg(mode, bound, fos, b2d)
    row, col = direction in ("both", "row"), direction in ("both", "col")
    g = gpu_quantize(x, c, rowwise=row, columnwise=col)
    o = oracle_quantize(x, c, rowwise=row, columnwise=col)
    what = f"case {i}: {rows}x{cols} {dtype} mode {mode} fos {fos} {bound} 2d {b2d} {direction}"
    for d in ("row", "col"):
        if d in g:
            assert_same(g[d], o[d], f"{what} {d}")


@pytest.mark.parametrize("i", range(24))
def test_random_transform_quantize_matches_oracle(i):
    rng = np.random.default_rng(3000 + i)
    rows = 16 * int(rng.integers(1, 40))
    dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float32
    step = 8 if dtype == torch.bfloat16 else 4  # 16-byte rows for the two-direction call
    cols = step * int(rng.integers(1, 120))
    mode = nv.NVFP4_ROW_SCALED if rng.random() < 0.6 else nv.NVFP4_PER_TENSOR
    fos = bool(rng.random() < 0.4)
    bound = 256.0 if (fos and rng.random() < 0.5) else 448.0
    mask = int(rng.integers(0, 1 << 16))
    x = workloads.seeded_normal(rows, cols, seed=4000 + i, dtype=dtype, device=DEV,
                                row_scale_decades=1.0)
    c = cfg(mode, bound, fos)
    rs = mode == nv.NVFP4_ROW_SCALED
    row = nv.alloc_out(rows, cols, rows if rs else 1, DEV)
    col = nv.alloc_out(cols, rows, cols if rs else 1, DEV)
    nv.nvfp4_quantize_both_rht(x, mask, c, row, col)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    kw = dict(mode=mode, bound=bound, four_over_six=fos)
    what = f"case {i}: {rows}x{cols} {dtype} mode {mode} fos {fos} {bound} mask {mask:#x}"
    assert_same(row, oracle.quantize(xb, tag, columnwise=False, **kw)["row"], f"{what} row")
    assert_same(col, oracle.quantize_columnwise_rht(xb, tag, mask, **kw), f"{what} col")
