"""Four-over-six on blocks whose two candidate errors are nearly or exactly equal,
compared byte for byte with the oracle.

The encode kernels first compare the two candidates ("Add NVFP4 four-over-six grouped
GEMM for MoE training", torchao PR #9, description: the block scaled to 4 or to 6 by
the lower squared error) through an estimate with a proven error bound, and compute
the exact in-order FP32 sums only for blocks the bound leaves open.  Random blocks
rarely come close to a tie, so these tests search for the closest ones: a CPU pass
computes both errors of every candidate block exactly as the dequantize formula
defines them ("Add backward overrides and 1x16 weights to NVFP4 four-over-six",
torchao PR #8, description) and keeps the blocks whose errors differ least relative
to D4^2 + D6^2 (the scale of the kernel's bound), together with every exact tie.
That search only picks inputs; the expected bytes come from the oracle.

Every row starts with an anchor block that holds the row's largest magnitude, so
that the line amax, and with it both dequantize factors, is the same in the search,
in the oracle and in the kernel, per tensor and row-scaled alike.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import assert_same, cfg, gpu_quantize, host_bits
from tests.test_kernel_fos_bound import candidate_errors

nv = pytest.importorskip("nvfp4_precision_quantization_gb300")

DEV = "cuda"
BLOCKS_PER_ROW = 64  # one anchor block + 63 selected blocks: rows of 1024 values
ANCHOR = 8.0


def _candidate_blocks(rng, n, dtype):
    """n blocks of 16 values below ANCHOR in magnitude, of mixed shapes."""
    scale = np.exp(rng.uniform(np.log(0.05), np.log(4.0), (n, 1)))
    x = rng.standard_normal((n, 16)) * scale
    heavy = rng.random(n) < 0.25  # a few blocks with one large value
    x[heavy, rng.integers(0, 16, heavy.sum())] *= 4.0
    ints = rng.random(n) < 0.1  # small integers and halves: exact ties are common
    x[ints] = rng.integers(-6, 7, (ints.sum(), 16)) * rng.choice([0.5, 1.0, 0.25], (ints.sum(), 1))
    x = np.clip(x, -ANCHOR * 0.99, ANCHOR * 0.99)
    if dtype == torch.bfloat16:
        return oracle.bf16_to_f32(oracle.f32_to_bf16(x.astype(np.float32))).astype(np.float32)
    return x.astype(np.float32)


def _near_tie_tensor(seed, bound, dtype, keep=63 * 64):
    """Rows of [anchor block | the `keep` candidate blocks closest to a tie]."""
    rng = np.random.default_rng(seed)
    cand = _candidate_blocks(rng, 300_000, dtype)
    c = candidate_errors(cand, np.full(len(cand), ANCHOR, np.float32), bound)
    err6, err4, D6, D4 = c[6]["err"], c[4]["err"], c[6]["D"], c[4]["D"]
    scale = D4.astype(np.float64) ** 2 + D6.astype(np.float64) ** 2
    rel = np.abs(err4.astype(np.float64) - err6) / scale
    ties = np.flatnonzero(rel == 0)[: keep // 4]  # exact ties: at most a quarter
    rest = np.flatnonzero(rel > 0)
    rest = rest[np.argsort(rel[rest], kind="stable")][: keep - len(ties)]
    order = np.concatenate([ties, rest])
    sel, rel_sel = cand[order], rel[order]
    rng.shuffle(sel)
    rows = keep // (BLOCKS_PER_ROW - 1)
    anchor = rng.standard_normal((rows, 16)).astype(np.float32)
    anchor = np.clip(anchor, -ANCHOR * 0.5, ANCHOR * 0.5)
    anchor[:, 5] = np.where(rng.random(rows) < 0.5, ANCHOR, -ANCHOR)
    x = np.concatenate([anchor[:, None, :], sel.reshape(rows, BLOCKS_PER_ROW - 1, 16)], axis=1)
    x = x.reshape(rows, BLOCKS_PER_ROW * 16)
    t = torch.from_numpy(x).to(dtype)
    assert float(t.float().abs().max()) == ANCHOR
    return t, rel_sel, (err4[order] < err6[order])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("bound", [256.0, 448.0])
def test_near_tie_search_reaches_the_bound(dtype, bound):
    """The selected blocks straddle the kernel's decision band (2^-12 of D4^2 + D6^2):
    many lie inside it (exact sums), many just outside (the bound decides), and both
    candidates win some of them."""
    _, rel, four_wins = _near_tie_tensor(11, bound, dtype)
    band = 2.0 ** -12
    assert (rel == 0).sum() >= 100
    assert ((rel > 0) & (rel < band)).sum() >= 100
    assert ((rel >= band) & (rel < 8 * band)).sum() >= 100
    assert 0 < four_wins.sum() < len(four_wins)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("bound", [256.0, 448.0])
@pytest.mark.parametrize("mode", ["row_scaled", "per_tensor"])
def test_near_ties_rowwise_and_both(dtype, bound, mode):
    m = nv.NVFP4_ROW_SCALED if mode == "row_scaled" else nv.NVFP4_PER_TENSOR
    x, _, _ = _near_tie_tensor(12, bound, dtype)
    x = x.to(DEV)
    c = cfg(m, bound, fos=True)
    xb, tag = host_bits(x)
    o = oracle.quantize(xb, tag, mode=m, bound=bound, four_over_six=True)
    g = gpu_quantize(x, c, columnwise=False)  # the rowwise-only kernel
    assert_same(g["row"], o["row"], "rowwise only")
    g = gpu_quantize(x, c)  # both directions in one kernel
    assert_same(g["row"], o["row"], "both: row")
    assert_same(g["col"], o["col"], "both: col")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("bound", [256.0, 448.0])
def test_near_ties_columnwise(dtype, bound):
    """The same blocks down the columns (x transposed): the columnwise-only kernel
    and the columnwise half of the two-direction kernel."""
    x, _, _ = _near_tie_tensor(13, bound, dtype)
    x = x.t().contiguous().to(DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, bound, fos=True)
    xb, tag = host_bits(x)
    o = oracle.quantize(xb, tag, mode=nv.NVFP4_ROW_SCALED, bound=bound, four_over_six=True)
    g = gpu_quantize(x, c, rowwise=False)
    assert_same(g["col"], o["col"], "columnwise only")
    g = gpu_quantize(x, c)
    assert_same(g["row"], o["row"], "both: row")
    assert_same(g["col"], o["col"], "both: col")
