"""Random Hadamard transform of the columnwise operand (GPU, through the C ABI)
against the oracle's reading R14 (TE-3206's description names the transform without
defining it): y = (1/4) H16 diag(s) x per column and 16-row block, FP32, bit for bit;
then the columnwise quantization of y, byte for byte."""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads
from gpu_helpers import assert_same, cfg, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _input(rows, cols, dtype, seed):
    return workloads.seeded_normal(rows, cols, seed=seed, dtype=dtype, device=DEV,
                                   row_scale_decades=1.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(16, 1), (64, 7), (128, 256), (2048, 200), (4096, 514)])
@pytest.mark.parametrize("mask", [0x0000, 0xFFFF, 0xBEEF])
def test_transform_matches_oracle_bit_for_bit(dtype, shape, mask):
    rows, cols = shape
    x = _input(rows, cols, dtype, seed=rows + cols)
    y = torch.full((rows, cols), float("nan"), dtype=torch.float32, device=DEV)
    nv.nvfp4_rht16(x, mask, y)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    exp = oracle.rht16(xb, tag, mask)
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), \
        f"{np.count_nonzero(got.view(np.uint32) != exp.view(np.uint32))} values differ"


def test_transform_in_place_and_unaligned_column_offset():
    x = _input(256, 130, torch.float32, seed=5)
    xb, _ = host_bits(x)
    exp = oracle.rht16(xb, "fp32", 0x1234)
    nv.nvfp4_rht16(x, 0x1234, x)  # in place (FP32 only)
    # a view that starts one column in: odd offset, so one column per thread
    base = _input(64, 33, torch.bfloat16, seed=6)
    sub = torch.empty(64, 32, dtype=torch.bfloat16, device=DEV)
    sub.copy_(base[:, 1:])
    y = torch.empty(64, 32, dtype=torch.float32, device=DEV)
    nv.nvfp4_rht16(sub, 0x00FF, y)
    torch.cuda.synchronize()
    assert np.array_equal(x.cpu().numpy().view(np.uint32), exp.view(np.uint32))
    sb, _ = host_bits(sub)
    assert np.array_equal(y.cpu().numpy().view(np.uint32),
                          oracle.rht16(sb, "bf16", 0x00FF).view(np.uint32))


# (mode, bound, four-over-six, 16x16 blocks); 1x16 blocks take the fused path (the
# amax and encode passes transform the blocks they read), 16x16 the workspace path
CONFIGS = [(nv.NVFP4_ROW_SCALED, 448.0, False, False), (nv.NVFP4_PER_TENSOR, 256.0, True, False),
           (nv.NVFP4_ROW_SCALED, 256.0, True, False), (nv.NVFP4_PER_TENSOR, 448.0, False, False),
           (nv.NVFP4_PER_TENSOR, 448.0, False, True), (nv.NVFP4_PER_TENSOR, 256.0, True, True)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
# (272, 40): a last tile of 16 rows; (16, 8): one block; (512, 75): odd columns
@pytest.mark.parametrize("shape", [(256, 200), (1024, 96), (4096, 130), (512, 75), (272, 40),
                                   (16, 8)])
@pytest.mark.parametrize("conf", CONFIGS)
def test_quantize_columnwise_rht_matches_oracle(dtype, shape, conf):
    rows, cols = shape
    x = _input(rows, cols, dtype, seed=11 + rows)
    c = cfg(*conf)
    mask = 0xA5C3
    col = nv.alloc_out(cols, rows, cols if conf[0] == nv.NVFP4_ROW_SCALED else 1, DEV)
    ws = torch.empty(rows * cols, dtype=torch.float32, device=DEV) if conf[3] else None
    nv.nvfp4_quantize_columnwise_rht(x, mask, c, col, ws)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    exp = oracle.quantize_columnwise_rht(xb, tag, mask, mode=conf[0], bound=conf[1],
                                         four_over_six=conf[2], block_2d=conf[3])
    assert_same(col, exp, f"rht {shape} {conf}")


def test_fused_equals_transform_then_quantize():
    """The fused call and the two-step composition of the public calls agree byte
    for byte (the transform into a buffer, then the plain columnwise quantize)."""
    x = _input(2048, 384, torch.bfloat16, seed=12)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    fused = nv.alloc_out(384, 2048, 384, DEV)
    nv.nvfp4_quantize_columnwise_rht(x, 0x0F0F, c, fused)
    y = torch.empty(2048, 384, dtype=torch.float32, device=DEV)
    nv.nvfp4_rht16(x, 0x0F0F, y)
    two = nv.alloc_out(384, 2048, 384, DEV)
    nv.nvfp4_quantize_columnwise(y, c, two)
    torch.cuda.synchronize()
    for a, b in ((fused.codes, two.codes), (fused.scales, two.scales), (fused.amax, two.amax)):
        assert torch.equal(a, b)


def test_full_size_sampled_columns():
    """The bench's operand (dY 16384 x 28672 BF16, row-scaled, bound 448) in the bench's
    launch configuration; 48 columns checked against the oracle (each column's result
    depends only on that column when the amax is per column)."""
    rows, cols = 16384, 28672
    x = workloads.linear(DEV)[1]  # dY of the linear-layer workload
    assert tuple(x.shape) == (rows, cols)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    col = nv.alloc_out(cols, rows, cols, DEV)
    nv.nvfp4_quantize_columnwise_rht(x, 0x6D2B, c, col)
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    pick = np.unique(np.concatenate([[0, 1, cols - 1], rng.integers(0, cols, 45)]))
    xs = x[:, torch.from_numpy(pick).to(DEV)].contiguous()
    xb, tag = host_bits(xs)
    exp = oracle.quantize_columnwise_rht(xb, tag, 0x6D2B, mode=nv.NVFP4_ROW_SCALED, bound=448.0)
    got = (col.codes[pick].cpu().numpy(), col.scales[pick].cpu().numpy(),
           col.amax[pick].cpu().numpy())
    assert np.array_equal(got[0], exp[0]) and np.array_equal(got[1], exp[1])
    assert np.array_equal(got[2].view(np.uint32), exp[2].view(np.uint32))


def test_noop_writes_nothing_and_empty_shapes():
    x = _input(64, 32, torch.bfloat16, seed=9)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    col = nv.alloc_out(32, 64, 32, DEV, fill=0xA5)
    col.amax.fill_(-1.0)
    ws = torch.full((64 * 32,), 3.0, dtype=torch.float32, device=DEV)
    noop = torch.ones(1, dtype=torch.float32, device=DEV)
    nv.nvfp4_quantize_columnwise_rht(x, 0x1, c, col, ws, noop=noop)  # fused path
    t = cfg(nv.NVFP4_PER_TENSOR, 448.0, False, True)  # 16x16: the workspace path
    col_t = nv.alloc_out(32, 64, 1, DEV, fill=0xA5)
    col_t.amax.fill_(-1.0)
    nv.nvfp4_quantize_columnwise_rht(x, 0x1, t, col_t, ws, noop=noop)
    torch.cuda.synchronize()
    for o in (col, col_t):
        assert bool((o.codes == 0xA5).all()) and bool((o.scales == 0xA5).all())
        assert bool((o.amax == -1.0).all())
    assert bool((ws == 3.0).all())
    # rows == 0: nothing to transform; the amax of the empty columns is 0
    e = torch.empty(0, 32, dtype=torch.bfloat16, device=DEV)
    col0 = nv.alloc_out(32, 0, 32, DEV)
    nv.nvfp4_quantize_columnwise_rht(e, 0x1, c, col0)
    torch.cuda.synchronize()
    assert bool((col0.amax == 0).all())


def test_rows_not_multiple_of_16_rejected():
    x = _input(40, 8, torch.bfloat16, seed=10)
    y = torch.empty(40, 8, dtype=torch.float32, device=DEV)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.nvfp4_rht16(x, 0, y)
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED


def test_given_amax_is_used_as_the_transform_amax():
    x = _input(512, 96, torch.bfloat16, seed=13)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    ref = nv.alloc_out(96, 512, 96, DEV)
    nv.nvfp4_quantize_columnwise_rht(x, 0x2468, c, ref)
    given = nv.alloc_out(96, 512, 96, DEV)
    given.amax_in = ref.amax.clone()
    nv.nvfp4_quantize_columnwise_rht(x, 0x2468, c, given)
    torch.cuda.synchronize()
    assert torch.equal(given.codes, ref.codes) and torch.equal(given.scales, ref.scales)
    assert torch.equal(given.amax, ref.amax)


def test_wgrad_gemm_on_transformed_operands():
    """The transform's use: dY and X quantized columnwise, both with the same signs,
    then dW = dY^T X on the tensor cores.  The result is within the GEMM's derived
    bound of the oracle's product of the same (oracle-made) operands.  Because the
    transform is orthonormal, it is also close to the unquantized dY^T X."""
    from test_gpu_gemm import _bound, _dev_op, _host_op
    rng = np.random.default_rng(14)
    tokens, d_out, d_in, mask = 512, 256, 192, 0x5A3C
    dy = (rng.standard_normal((tokens, d_out)) * np.exp(rng.uniform(-1, 1, (tokens, 1))))
    x = rng.standard_normal((tokens, d_in)) * 0.5
    dy_t = torch.from_numpy(dy.astype(np.float32)).to(DEV).to(torch.bfloat16)
    x_t = torch.from_numpy(x.astype(np.float32)).to(DEV).to(torch.bfloat16)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    ops, hosts = [], []
    for t, lines in ((dy_t, d_out), (x_t, d_in)):
        o = nv.alloc_out(lines, tokens, lines, DEV)
        nv.nvfp4_quantize_columnwise_rht(t, mask, c, o)
        ops.append(o.as_operand(nv.NVFP4_ROW_SCALED, 448.0))
        tb, tag = host_bits(t)
        hosts.append(_host_op(*oracle.quantize_columnwise_rht(tb, tag, mask), nv.NVFP4_ROW_SCALED,
                              448.0))
    d = torch.empty(d_out, d_in, dtype=torch.float32, device=DEV)
    nv.nvfp4_gemm(ops[0], ops[1], d)
    torch.cuda.synchronize()
    # the GPU's quantized operands are the oracle's, byte for byte
    for o, h in zip(ops, hosts):
        assert np.array_equal(o.codes.cpu().numpy(), h["codes"])
    exact, dabs = oracle.gemm(hosts[0], hosts[1], with_abs=True)
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - exact) <= _bound(tokens, dabs, exact, False))
    ref = dy_t.float().cpu().numpy().astype(np.float64).T @ x_t.float().cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - ref) < 0.2 * np.linalg.norm(ref)


# ---------------------------------------------------------------- both directions

def _both_expected(x, mask, conf, parallel=False):
    """Rowwise quantization of x and columnwise quantization of its transform, each
    from the oracle on its own."""
    xb, tag = host_bits(x)
    kw = dict(mode=conf[0], bound=conf[1], four_over_six=conf[2])
    if parallel:
        row = oracle.quantize_parallel(xb, tag, columnwise=False, **kw)["row"]
        col = oracle.quantize_parallel(oracle.rht16(xb, tag, mask), "fp32", rowwise=False,
                                       **kw)["col"]
    else:
        row = oracle.quantize(xb, tag, columnwise=False, **kw)["row"]
        col = oracle.quantize_columnwise_rht(xb, tag, mask, **kw)
    return row, col


def _both_gpu(x, mask, conf, noop=None, fill=None, amax_in=(None, None)):
    rows, cols = x.shape
    rs = conf[0] == nv.NVFP4_ROW_SCALED
    row = nv.alloc_out(rows, cols, rows if rs else 1, DEV, fill)
    col = nv.alloc_out(cols, rows, cols if rs else 1, DEV, fill)
    row.amax_in, col.amax_in = amax_in
    nv.nvfp4_quantize_both_rht(x, mask, cfg(*conf), row, col, noop=noop)
    torch.cuda.synchronize()
    return row, col


BOTH_CONFIGS = [c for c in CONFIGS if not c[3]]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
# (512, 1024), (256, 256): code pitches multiples of 32 bytes (BF16: sector stores);
# (2048, 384): 16 but not 32 (direct stores); (272, 40): a last tile of 16 rows;
# (16, 8): one block.  Where the column pairs fill whole CTAs (512, 1024, 3584 BF16
# columns...) one read of x gives both maxima: (512, 1024), (272, 512) and (400, 1024)
# take that path, the last two with a partial last run of row blocks.
@pytest.mark.parametrize("shape", [(512, 1024), (256, 256), (2048, 384), (272, 40), (16, 8),
                                   (1024, 96), (272, 512), (400, 1024)])
@pytest.mark.parametrize("conf", BOTH_CONFIGS)
def test_quantize_both_rht_matches_oracle(dtype, shape, conf):
    """Both directions in one call (one encode pass, or one per direction with
    four-over-six), the transform on the columnwise side only
    ("NVFP4: enable row-scaled transpose quantization for backward", TE PR #3206,
    description: rowwise for fprop, the transposed operand for wgrad)."""
    rows, cols = shape
    x = _input(rows, cols, dtype, seed=31 + rows + cols)
    mask = 0x5A3C
    row, col = _both_gpu(x, mask, conf)
    er, ec = _both_expected(x, mask, conf)
    assert_same(row, er, f"both-rht row {shape} {conf}")
    assert_same(col, ec, f"both-rht col {shape} {conf}")


@pytest.mark.parametrize("conf", BOTH_CONFIGS)
def test_quantize_both_rht_multitile(conf):
    """4096 x 4096 BF16 (1024 tiles, several per CTA, sector stores) and 2048 x 3000
    FP32 (direct stores), compared in full with the oracle run in host threads."""
    for x in (workloads.outliers(DEV), _input(2048, 3000, torch.float32, seed=41)):
        row, col = _both_gpu(x, 0x6D2B, conf)
        er, ec = _both_expected(x, 0x6D2B, conf, parallel=True)
        assert_same(row, er, f"both-rht row {tuple(x.shape)} {conf}")
        assert_same(col, ec, f"both-rht col {tuple(x.shape)} {conf}")


def test_quantize_both_rht_equals_the_two_calls():
    """The one-pass call gives the bytes of the rowwise quantize of x and the fused
    columnwise quantize of its transform, called separately."""
    x = _input(2048, 3584, torch.bfloat16, seed=42)
    for conf in BOTH_CONFIGS:
        c = cfg(*conf)
        rs = conf[0] == nv.NVFP4_ROW_SCALED
        row, col = _both_gpu(x, 0x0F0F, conf)
        r2 = nv.alloc_out(2048, 3584, 2048 if rs else 1, DEV)
        nv.nvfp4_quantize_rowwise(x, c, r2)
        c2 = nv.alloc_out(3584, 2048, 3584 if rs else 1, DEV)
        nv.nvfp4_quantize_columnwise_rht(x, 0x0F0F, c, c2)
        torch.cuda.synchronize()
        for a, b in ((row, r2), (col, c2)):
            assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            assert torch.equal(a.amax, b.amax)


def test_quantize_both_rht_given_amax_and_noop():
    x = _input(512, 256, torch.bfloat16, seed=43)
    conf = (nv.NVFP4_PER_TENSOR, 448.0, False, False)
    ref_r, ref_c = _both_gpu(x, 0x2468, conf)
    # given maxima: the row one is x's, the column one the transform's
    row, col = _both_gpu(x, 0x2468, conf, amax_in=(ref_r.amax.clone(), ref_c.amax.clone()))
    for a, b in ((row, ref_r), (col, ref_c)):
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
        assert torch.equal(a.amax, b.amax)
    assert not torch.equal(ref_r.amax, ref_c.amax)  # two different tensors
    noop = torch.ones(1, dtype=torch.float32, device=DEV)
    # (256, 1024): the one-read amax of both maxima; (512, 256): the two passes
    for xx in (x, _input(256, 1024, torch.bfloat16, seed=44)):
        for cf in (conf, (nv.NVFP4_ROW_SCALED, 448.0, False, False)):
            row, col = _both_gpu(xx, 0x2468, cf, noop=noop, fill=0xA5)
            for o in (row, col):
                assert bool((o.codes == 0xA5).all()) and bool((o.scales == 0xA5).all())
    # empty shapes: no rows (each column's amax is 0), no columns
    for rows, cols in ((0, 64), (32, 0)):
        e = torch.empty(rows, cols, dtype=torch.bfloat16, device=DEV)
        r0, c0 = _both_gpu(e, 0x1, (nv.NVFP4_ROW_SCALED, 448.0, False, False))
        assert bool((r0.amax == 0).all()) and bool((c0.amax == 0).all())
    # only one maximum given: the other is computed on its own
    x2 = _input(256, 1024, torch.bfloat16, seed=45)
    ref_r, ref_c = _both_gpu(x2, 0x1357, conf)
    for given in ((ref_r.amax.clone(), None), (None, ref_c.amax.clone())):
        row, col = _both_gpu(x2, 0x1357, conf, amax_in=given)
        for a, b in ((row, ref_r), (col, ref_c)):
            assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            assert torch.equal(a.amax, b.amax)
