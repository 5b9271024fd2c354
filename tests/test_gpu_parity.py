"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, byte
for byte -- codes, E4M3 scales, amax bit patterns, dequantized values.

Sizes span several 128-row tiles with ragged tails; the workload-sized cases
live in test_gpu_workloads.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_same, cfg, gpu_quantize, host_bits, oracle_quantize

nv = pytest.importorskip("nvfp4_precision_quantization_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda"

SHAPES = [(256, 256), (300, 200), (130, 1000), (1, 16), (17, 33), (129, 257), (512, 384),
          (272, 400), (264, 512), (136, 224)]


def _x(shape, dtype, seed, decades=2.0):
    return workloads.seeded_normal(*shape, seed=seed, dtype=dtype, device="cpu",
                                   row_scale_decades=decades).to(DEV)


# ---------------------------------------------------------------- conversions

def _conversion_inputs():
    parts = [(np.arange(65536, dtype=np.uint32) << 16).view(np.float32)]
    for v in [0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0, 7.0, 8.0]:
        b = int(np.array([v], np.float32).view(np.int32)[0])
        k = np.arange(b - 4096, b + 4097, dtype=np.int64).astype(np.uint32)
        parts.append(k.view(np.float32))
    grid = np.array([oracle.lib().oracle_e4m3_decode(k) for k in range(1, 0x7F)], np.float32)
    mids = ((grid[:-1].astype(np.float64) + grid[1:]) / 2).astype(np.float32)
    for v in np.concatenate([grid, mids, [464.0, 480.0, 2.0**-10]]).astype(np.float32):
        b = int(np.array([v], np.float32).view(np.int32)[0])
        parts.append(np.arange(b - 64, b + 65, dtype=np.int64).astype(np.uint32).view(np.float32))
    rng = np.random.default_rng(0)
    parts.append(rng.integers(0, 2**32, 4_000_000, dtype=np.uint64).astype(np.uint32)
                 .view(np.float32))
    x = np.concatenate(parts)
    x = np.concatenate([x, -x])
    return x[~np.isnan(x)]


def test_device_conversions_match_oracle():
    x = _conversion_inputs()
    xt = torch.from_numpy(x).to(DEV)
    e2 = torch.empty(x.size, dtype=torch.uint8, device=DEV)
    e4 = torch.empty(x.size, dtype=torch.uint8, device=DEV)
    nv.nvfp4_selftest_convert(xt, e2, e4)
    g2, g4 = e2.cpu().numpy(), e4.cpu().numpy()
    r2 = oracle.e2m1_encode(x)
    bad = np.nonzero(g2 != r2)[0]
    assert bad.size == 0, ("e2m1", x[bad[:8]], g2[bad[:8]], r2[bad[:8]])
    # the E4M3 oracle is a linear search: check a strided subset plus all small values
    sel = np.concatenate([np.arange(0, x.size, 7), np.nonzero(np.abs(x) < 600)[0][::3]])
    r4 = oracle.e4m3_encode(x[sel])
    bad = np.nonzero(g4[sel] != r4)[0]
    assert bad.size == 0, ("e4m3", x[sel][bad[:8]], g4[sel][bad[:8]], r4[bad[:8]])


def test_nibble_order():
    x = torch.tensor([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -6.0], device=DEV)
    e2 = torch.empty(9, dtype=torch.uint8, device=DEV)
    nv.nvfp4_selftest_convert(x, e2, None)
    assert e2.cpu().tolist() == [1, 2, 3, 4, 5, 6, 7, 9, 15]


# ---------------------------------------------------------------- amax

@pytest.mark.parametrize("shape", SHAPES + [(4000, 5000)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_amax_matches_oracle(shape, dtype):
    x = _x(shape, dtype, seed=1, decades=3)
    r = torch.empty(shape[0], device=DEV)
    c = torch.empty(shape[1], device=DEV)
    t = torch.empty(1, device=DEV)
    nv.nvfp4_amax(x, r, c, t)
    xb, tag = host_bits(x)
    ra, ca, ta = oracle.amax(xb, tag)
    assert np.array_equal(r.cpu().numpy().view(np.uint32), ra.view(np.uint32))
    assert np.array_equal(c.cpu().numpy().view(np.uint32), ca.view(np.uint32))
    assert t.item() == ta


def test_amax_each_output_alone():
    x = _x((300, 520), torch.bfloat16, seed=2)
    xb, tag = host_bits(x)
    ra, ca, ta = oracle.amax(xb, tag)
    r = torch.empty(300, device=DEV)
    nv.nvfp4_amax(x, row_amax=r)
    c = torch.empty(520, device=DEV)
    nv.nvfp4_amax(x, col_amax=c)
    t = torch.empty(1, device=DEV)
    nv.nvfp4_amax(x, tensor_amax=t)
    assert np.array_equal(r.cpu().numpy(), ra) and np.array_equal(c.cpu().numpy(), ca)
    assert t.item() == ta


# ---------------------------------------------------------------- quantize

@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("fos,bound", [(False, 448.0), (True, 256.0), (True, 448.0)])
def test_quantize_both_matches_oracle(shape, dtype, mode, fos, bound):
    x = _x(shape, dtype, seed=3)
    c = cfg(mode, bound, fos)
    g = gpu_quantize(x, c)
    o = oracle_quantize(x, c)
    assert_same(g["row"], o["row"], "row")
    assert_same(g["col"], o["col"], "col")


@pytest.mark.parametrize("direction", ["row", "col"])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
def test_quantize_single_direction(direction, mode):
    x = _x((333, 264), torch.bfloat16, seed=4)
    c = cfg(mode)
    g = gpu_quantize(x, c, rowwise=direction == "row", columnwise=direction == "col")
    o = oracle_quantize(x, c, rowwise=direction == "row", columnwise=direction == "col")
    assert_same(g[direction], o[direction], direction)


@pytest.mark.parametrize("shape", [(256, 256), (300, 200), (64, 1000), (33, 48)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fos", [False, True])
def test_quantize_2d_blocks_matches_oracle(shape, dtype, fos):
    x = _x(shape, dtype, seed=5, decades=0)
    c = cfg(nv.NVFP4_PER_TENSOR, 448.0, fos, b2d=True)
    g = gpu_quantize(x, c)
    o = oracle_quantize(x, c)
    assert_same(g["row"], o["row"], "row")
    assert_same(g["col"], o["col"], "col")


def test_quantize_with_given_amax():
    x = _x((200, 300), torch.bfloat16, seed=6)
    xb, tag = host_bits(x)
    ra, ca, _ = oracle.amax(xb, tag)
    ra = ra * np.float32(1.5)   # any positive amax is allowed
    ca = ca * np.float32(0.75)
    # four-over-six too: both directions then run as one pass per direction
    for fos in (False, True):
        c = cfg(nv.NVFP4_ROW_SCALED, 448.0, fos)
        g = gpu_quantize(x, c, row_amax_in=torch.from_numpy(ra).to(DEV),
                         col_amax_in=torch.from_numpy(ca).to(DEV))
        o = oracle_quantize(x, c, row_amax_in=ra, col_amax_in=ca)
        assert_same(g["row"], o["row"], f"row fos={fos}")
        assert_same(g["col"], o["col"], f"col fos={fos}")
    # per-tensor with different scalars per direction, 16x16 blocks too
    for b2d, fos in ((False, False), (True, False), (False, True), (True, True)):
        c = cfg(nv.NVFP4_PER_TENSOR, 448.0, fos, b2d)
        g = gpu_quantize(x, c, row_amax_in=torch.tensor([7.0], device=DEV),
                         col_amax_in=torch.tensor([3.0], device=DEV))
        o = oracle_quantize(x, c, row_amax_in=np.array([7.0], np.float32),
                            col_amax_in=np.array([3.0], np.float32))
        assert_same(g["row"], o["row"], f"row b2d={b2d} fos={fos}")
        assert_same(g["col"], o["col"], f"col b2d={b2d} fos={fos}")


def test_zero_rows_and_zero_tensor():
    x = workloads.edge_zero_rows(512, 384, device="cpu").to(DEV)
    for mode in (nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR):
        c = cfg(mode)
        g, o = gpu_quantize(x, c), oracle_quantize(x, c)
        assert_same(g["row"], o["row"]), assert_same(g["col"], o["col"])
    z = torch.zeros(300, 200, dtype=torch.bfloat16, device=DEV)
    for mode in (nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR):
        g = gpu_quantize(z, cfg(mode), fill=0xA5)
        for d in ("row", "col"):
            assert not g[d].codes.any() and not g[d].scales.any() and not g[d].amax.any()


def test_noop_preserves_everything():
    x = _x((300, 260), torch.bfloat16, seed=7)
    flag = torch.ones(1, device=DEV)
    for mode in (nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR):
        for fos in (False, True):  # four-over-six: one encode pass per direction
            g = gpu_quantize(x, cfg(mode, 448.0, fos), noop=flag, fill=0xA5,
                             outs={"row": nv.alloc_out(300, 260, 300 if mode else 1, DEV, 0xA5),
                                   "col": nv.alloc_out(260, 300, 260 if mode else 1, DEV, 0xA5)})
            for d in ("row", "col"):
                g[d].amax.fill_(-1.0)
            g = gpu_quantize(x, cfg(mode, 448.0, fos), noop=flag, outs=g)
            for d in ("row", "col"):
                assert torch.all(g[d].codes == 0xA5) and torch.all(g[d].scales == 0xA5)
                assert torch.all(g[d].amax == -1.0)
    # amax entry point and grouped entry points too
    r = torch.full((300,), -1.0, device=DEV)
    nv.nvfp4_amax(x, row_amax=r, noop=flag)
    assert torch.all(r == -1.0)
    ends = torch.tensor([100, 300], dtype=torch.int64, device=DEV)
    ga = torch.full((2,), -1.0, device=DEV)
    out = nv.alloc_out(300, 260, 300, DEV, 0xA5)
    out.amax.fill_(-1.0)
    nv.nvfp4_grouped_quantize_rowwise(x, ends, cfg(nv.NVFP4_PER_TENSOR, 256.0, True), out, ga,
                                      noop=flag)
    torch.cuda.synchronize()
    assert torch.all(ga == -1.0) and torch.all(out.amax == -1.0) and torch.all(out.codes == 0xA5)
    # flag 0 means run
    g = gpu_quantize(x, cfg(), noop=torch.zeros(1, device=DEV))
    assert_same(g["row"], oracle_quantize(x, cfg())["row"])


def test_empty_inputs():
    for shape in ((0, 64), (64, 0), (0, 0)):
        x = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
        g = gpu_quantize(x, cfg(nv.NVFP4_ROW_SCALED), fill=0)
        assert g["row"].amax.numel() == shape[0] and g["col"].amax.numel() == shape[1]
        assert not g["row"].amax.any() and not g["col"].amax.any()
        g = gpu_quantize(x, cfg(nv.NVFP4_PER_TENSOR))
        assert g["row"].amax.item() == 0.0 and g["col"].amax.item() == 0.0


def test_non_default_stream():
    x = _x((256, 512), torch.bfloat16, seed=8)
    s = torch.cuda.Stream()
    c = cfg()
    outs = {"row": nv.alloc_out(256, 512, 256, DEV), "col": nv.alloc_out(512, 256, 512, DEV)}
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        nv.nvfp4_quantize_both(x, c, outs["row"], outs["col"])
    s.synchronize()
    o = oracle_quantize(x, c)
    assert_same(outs["row"], o["row"]), assert_same(outs["col"], o["col"])


def test_misaligned_input_uses_plain_loads():
    # a view whose base is not 16-byte aligned: TMA cannot be used
    big = _x((64, 129), torch.bfloat16, seed=9)
    x = big.view(-1)[1:1 + 64 * 128].view(64, 128)
    assert x.data_ptr() % 16 != 0
    c = cfg()
    g, o = gpu_quantize(x, c), oracle_quantize(x, c)
    assert_same(g["row"], o["row"]), assert_same(g["col"], o["col"])


# ---------------------------------------------------------------- dequantize

@pytest.mark.parametrize("shape", [(256, 256), (300, 200), (33, 17)])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("bound", [448.0, 256.0])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_dequantize_matches_oracle(shape, mode, bound, out_dtype):
    x = _x(shape, torch.bfloat16, seed=10)
    xb, tag = host_bits(x)
    q = oracle.quantize(xb, tag, mode=mode, bound=bound, columnwise=False)["row"]
    rows, cols = shape
    out = torch.empty(shape, dtype=out_dtype, device=DEV)
    nv.nvfp4_dequantize(torch.from_numpy(q[0]).to(DEV), torch.from_numpy(q[1]).to(DEV),
                        torch.from_numpy(q[2]).to(DEV), mode, rows, cols, bound, out)
    ref = oracle.dequantize(q[0], q[1], q[2], row_scaled=mode == nv.NVFP4_ROW_SCALED, rows=rows,
                            cols=cols, bound=bound,
                            out_dtype="bf16" if out_dtype == torch.bfloat16 else "fp32")
    got = out.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if out_dtype == torch.bfloat16 \
        else got.numpy().view(np.uint32)
    assert np.array_equal(got, ref.view(got.dtype))


# ---------------------------------------------------------------- grouped

def _groups(counts, cols, align, seed):
    padded = [-(-n // align) * align for n in counts]
    ends = np.cumsum(padded).astype(np.int64)
    x = torch.zeros(int(ends[-1]), cols, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(seed)
    start = 0
    for n, p in zip(counts, padded):
        x[start:start + n] = (torch.randn(n, cols, generator=g) * (1 + 3 * torch.rand(1, generator=g))).to(torch.bfloat16)
        start += p
    return x.to(DEV), ends


@pytest.mark.parametrize("mode", [nv.NVFP4_PER_TENSOR, nv.NVFP4_ROW_SCALED])
@pytest.mark.parametrize("fos,bound", [(True, 256.0), (False, 448.0)])
def test_grouped_quantize_matches_oracle(mode, fos, bound):
    x, ends = _groups([5, 0, 130, 37, 300, 1], 512, 128, seed=11)
    rows, cols = x.shape
    ga = torch.empty(len(ends), device=DEV)
    out = nv.alloc_out(rows, cols, rows, DEV)
    nv.nvfp4_grouped_quantize_rowwise(x, torch.from_numpy(ends).to(DEV), cfg(mode, bound, fos),
                                      out, ga)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    codes, scales, ra, gam = oracle.grouped_quantize_rowwise(xb, tag, ends, mode=mode,
                                                              bound=bound, four_over_six=fos)
    assert_same(out, (codes, scales, ra), "grouped")
    assert np.array_equal(ga.cpu().numpy(), gam)


def test_grouped_amax_matches_oracle():
    x, ends = _groups([7, 128, 0, 250], 384, 1, seed=12)
    ga = torch.empty(len(ends), device=DEV)
    ex = torch.empty(x.shape[0], device=DEV)
    nv.nvfp4_grouped_amax(x, torch.from_numpy(ends).to(DEV), ga, ex)
    xb, tag = host_bits(x)
    g, e = oracle.grouped_amax(xb, tag, ends)
    assert np.array_equal(ga.cpu().numpy(), g) and np.array_equal(ex.cpu().numpy(), e)


@pytest.mark.parametrize("with_rows", [True, False])
def test_grouped_amax_many_groups(with_rows):
    """1000 groups (empty ones included), more than the reduction's CTAs: each CTA
    takes several groups.  With the per-row output the maxima come from the tiled row
    pass and the per-group reduction, without it from the grouped kernel."""
    rng = np.random.default_rng(15)
    counts = rng.integers(0, 24, 1000).tolist()
    counts[3] = 0
    x, ends = _groups(counts, 200, 1, seed=16)
    ga = torch.full((len(ends),), -1.0, device=DEV)
    ex = torch.full((x.shape[0],), -1.0, device=DEV) if with_rows else None
    nv.nvfp4_grouped_amax(x, torch.from_numpy(ends).to(DEV), ga, ex)
    xb, tag = host_bits(x)
    g, e = oracle.grouped_amax(xb, tag, ends)
    assert np.array_equal(ga.cpu().numpy(), g)
    if with_rows:
        assert np.array_equal(ex.cpu().numpy(), e)


def test_grouped_invalid_ends_write_nothing_and_set_status():
    x, _ = _groups([64, 64], 256, 1, seed=13)
    nv.nvfp4_device_status(reset=True)
    bad = torch.tensor([100, 60], dtype=torch.int64, device=DEV)
    ga = torch.full((2,), -1.0, device=DEV)
    out = nv.alloc_out(128, 256, 128, DEV, 0xA5)
    out.amax.fill_(-1.0)
    nv.nvfp4_grouped_quantize_rowwise(x, bad, cfg(nv.NVFP4_PER_TENSOR, 256.0, True), out, ga)
    assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS
    assert torch.all(ga == -1.0) and torch.all(out.amax == -1.0)
    assert torch.all(out.codes == 0xA5) and torch.all(out.scales == 0xA5)
    assert nv.nvfp4_device_status() == 0



@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fos,bound", [(True, 256.0), (False, 448.0)])
@pytest.mark.parametrize("counts,cols", [
    ([100, 156, 0, 300, 212], 640),   # ends 100, 256, 256, 556, 768
    ([77, 300, 135], 300),            # no end on a tile boundary but the last
    ([256] * 40, 1024),               # 40 groups, several tiles per CTA
    ([128, 0, 0, 128], 128),          # empty groups
])
def test_grouped_quantize_per_group_amax_any_ends(dtype, fos, bound, counts, cols):
    """Per-group amax, rowwise, with rows a multiple of 128 and group ends anywhere
    (inside tiles, on tile boundaries, empty groups, many groups): the row maxima,
    each group's maximum over its rows and the encode with each row's group amax."""
    x, ends = _groups(counts, cols, 1, seed=14)
    x = x.to(dtype)
    rows = x.shape[0]
    assert rows % 128 == 0
    ga = torch.full((len(ends),), -1.0, device=DEV)
    out = nv.alloc_out(rows, cols, rows, DEV, 0xA5)
    out.amax.fill_(-1.0)
    nv.nvfp4_grouped_quantize_rowwise(x, torch.from_numpy(ends).to(DEV),
                                      cfg(nv.NVFP4_PER_TENSOR, bound, fos), out, ga)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    codes, scales, ra, gam = oracle.grouped_quantize_rowwise(xb, tag, ends, mode=nv.NVFP4_PER_TENSOR,
                                                              bound=bound, four_over_six=fos)
    assert_same(out, (codes, scales, ra), "grouped")
    assert np.array_equal(ga.cpu().numpy(), gam)
    assert nv.nvfp4_device_status() == 0


@pytest.mark.parametrize("shape", [(256, 256), (640, 300), (4096, 2048)])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("fos,bound", [(False, 448.0), (True, 256.0)])
def test_quantize_columnwise_only_sector_stores(shape, mode, fos, bound):
    """Columnwise only, BF16, rows a multiple of 64: lane pairs exchange their 32-row
    halves and store each column's codes as whole 32-byte sectors (4096 x 2048: 512
    tiles, so CTAs walk several)."""
    x = _x(shape, torch.bfloat16, seed=15)
    c = cfg(mode, bound, fos)
    g = gpu_quantize(x, c, rowwise=False)
    o = oracle_quantize(x, c, rowwise=False)
    assert_same(g["col"], o["col"], "col")
