"""GPU parity on the workload shapes (see workloads.py), in the launch
configuration the benchmark times.

Small workloads are compared in full.  The large ones (the 16384 x 8192 /
16384 x 28672 linear-layer operands, the 65536-token MoE tensor, the 8192 x 8192
16x16 case) are compared on sampled rows and columns that the oracle computes
one line at a time from the same bytes, plus properties that hold at any size.
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


def _line_f32(t: torch.Tensor) -> np.ndarray:
    b, tag = host_bits(t.reshape(1, -1))
    return oracle.as_f32(b, tag).reshape(-1)


def _check_sampled_rows(x, out, rows_idx, amax_of, bound=448.0, fos=False):
    codes = out.codes[rows_idx].cpu().numpy()
    scales = out.scales[rows_idx].cpu().numpy()
    amax = out.amax[rows_idx].cpu().numpy()
    for i, r in enumerate(rows_idx.tolist()):
        v = _line_f32(x[r])
        a = amax_of(r, v)
        c, s = oracle.quantize_line(v, a, bound, fos)
        assert amax[i] == a, (r, amax[i], a)
        assert np.array_equal(codes[i], c), r
        assert np.array_equal(scales[i], s), r


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)])))


def test_tiny_full():
    x = workloads.tiny(DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0)
    g, o = gpu_quantize(x, c), oracle_quantize(x, c)
    assert_same(g["row"], o["row"], "row")
    assert_same(g["col"], o["col"], "col")


@pytest.mark.parametrize("mode", [nv.NVFP4_PER_TENSOR, nv.NVFP4_ROW_SCALED])
def test_outliers_full_with_dequantize(mode):
    x = workloads.outliers(DEV)
    c = cfg(mode, 448.0)
    g, o = gpu_quantize(x, c), oracle_quantize(x, c)
    assert_same(g["row"], o["row"], "row")
    assert_same(g["col"], o["col"], "col")
    rows, cols = x.shape
    for od, tag in ((torch.bfloat16, "bf16"), (torch.float32, "fp32")):
        out = torch.empty(rows, cols, dtype=od, device=DEV)
        nv.nvfp4_dequantize(g["row"].codes, g["row"].scales, g["row"].amax, mode, rows, cols,
                            448.0, out)
        ref = oracle.dequantize(o["row"][0], o["row"][1], o["row"][2],
                                row_scaled=mode == nv.NVFP4_ROW_SCALED, rows=rows, cols=cols,
                                out_dtype=tag)
        got = out.cpu()
        got = got.view(torch.int16).numpy().view(np.uint16) if tag == "bf16" \
            else got.numpy().view(np.uint32)
        assert np.array_equal(got, ref.view(got.dtype))


@pytest.fixture(scope="module")
def linear_operands():
    x, dy = workloads.linear(DEV)
    out = {}
    for name, t in (("x", x), ("dy", dy)):
        xb, tag = host_bits(t)
        out[name] = (t, oracle.amax(xb, tag))  # the oracle's full row / column / tensor amax
    return out


def _check_sampled_lines(x, g, ri, ci, mode, amaxes, bound=448.0, fos=False):
    """Sampled rows of the rowwise output and sampled columns of the columnwise output
    against the oracle, one line at a time from the same bytes."""
    ra, ca, t = amaxes
    rs = mode == nv.NVFP4_ROW_SCALED
    _check_sampled_rows(x, g["row"] if rs else _per_line(g["row"], ri),
                        ri, lambda r, v: ra[r] if rs else np.float32(t), bound, fos)
    xt_cols = x[:, ci.to(DEV)].t().contiguous()
    gc = g["col"]
    codes = gc.codes[ci].cpu().numpy()
    scales = gc.scales[ci].cpu().numpy()
    for i, c in enumerate(ci.tolist()):
        v = _line_f32(xt_cols[i])
        a = ca[c] if rs else np.float32(t)
        cc, ss = oracle.quantize_line(v, a, bound, fos)
        assert np.array_equal(codes[i], cc), ("col codes", c)
        assert np.array_equal(scales[i], ss), ("col scales", c)
    if rs:
        assert np.array_equal(gc.amax.cpu().numpy(), ca)
    else:
        assert g["row"].amax.item() == t and gc.amax.item() == t


def _per_line(out, ri):
    """A per-tensor output seen through the row checker: its one amax repeated."""
    return nv.Out(out.codes, out.scales, out.amax.expand(out.codes.shape[0]))


@pytest.mark.parametrize("which", ["x", "dy"])
def test_linear_operands_sampled(linear_operands, which):
    x, amaxes = linear_operands[which]
    rows, cols = x.shape
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0)
    g = gpu_quantize(x, c)
    ri = _sample(rows, 40, 1)
    ci = _sample(cols, 40, 2)
    _check_sampled_lines(x, g, ri, ci, nv.NVFP4_ROW_SCALED, amaxes)
    # the full amax vectors against the oracle's reduction of the whole matrix
    assert np.array_equal(g["row"].amax.cpu().numpy(), amaxes[0])
    assert np.array_equal(g["col"].amax.cpu().numpy(), amaxes[1])
    # property at any size: every row's block holding the row amax has scale 0x7E
    top = (g["row"].scales == 0x7E).any(dim=1)
    assert bool(top[g["row"].amax > 0].all())


@pytest.mark.parametrize("which", ["x", "dy"])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("bound", [256.0, 448.0])
def test_linear_operands_fos_sampled(linear_operands, which, mode, bound):
    """Four-over-six on the linear-layer operands, both directions: the configuration
    of the four-over-six benchmark row, each CTA walking 13 (X) or 47 (dY) tiles."""
    x, amaxes = linear_operands[which]
    rows, cols = x.shape
    g = gpu_quantize(x, cfg(mode, bound, fos=True))
    _check_sampled_lines(x, g, _sample(rows, 32, 5), _sample(cols, 32, 6), mode, amaxes,
                         bound=bound, fos=True)


@pytest.fixture(scope="module")
def moe_operands():
    return workloads.moe(DEV)


def test_moe_grouped_sampled(moe_operands):
    x, ends, counts, padded = moe_operands
    rows, cols = x.shape
    c = cfg(nv.NVFP4_PER_TENSOR, 256.0, fos=True)
    ga = torch.empty(len(ends), device=DEV)
    out = nv.alloc_out(rows, cols, rows, DEV)
    nv.nvfp4_grouped_quantize_rowwise(x, ends, c, out, ga)
    torch.cuda.synchronize()
    xb, tag = host_bits(x)
    ends_np = ends.cpu().numpy()
    gam, exp = oracle.grouped_amax(xb, tag, ends_np)
    assert np.array_equal(ga.cpu().numpy(), gam)
    assert np.array_equal(out.amax.cpu().numpy(), exp)
    starts = np.concatenate([[0], ends_np[:-1]])
    ri = _sample(rows, 48, 3)
    # also the first padding row of a few groups
    pads = [int(s + n) for s, n, p in zip(starts, counts.tolist(), padded.tolist()) if n < p][:8]
    ri = torch.unique(torch.cat([ri, torch.tensor(pads, dtype=ri.dtype)]))
    grp = np.searchsorted(ends_np, ri.numpy(), side="right")
    _check_sampled_rows(x, out, ri, lambda r, v: gam[grp[list(ri.tolist()).index(r)]],
                        bound=256.0, fos=True)
    pad_rows = torch.tensor(pads, dtype=torch.long)
    assert not out.codes[pad_rows].any() and not out.scales[pad_rows].any()


def test_moe_ragged_padded_equals_aligned(moe_operands):
    x, ends, counts, padded = moe_operands
    xr, ends_r = workloads.moe_ragged(x, counts, padded)
    c = cfg(nv.NVFP4_PER_TENSOR, 256.0, fos=True)
    outs = []
    for xx, ee in ((x, ends), (xr.contiguous(), ends_r.to(DEV))):
        o = nv.alloc_out(xx.shape[0], xx.shape[1], xx.shape[0], DEV)
        nv.nvfp4_grouped_quantize_rowwise(xx, ee, c, o, torch.empty(len(ee), device=DEV))
        outs.append(o)
    torch.cuda.synchronize()
    keep = torch.cat([torch.arange(int(s), int(s) + int(n)) for s, n in
                      zip(torch.cat([torch.zeros(1, dtype=torch.int64), ends.cpu()[:-1]]), counts)])
    assert torch.equal(outs[0].codes[keep.to(DEV)], outs[1].codes)
    assert torch.equal(outs[0].scales[keep.to(DEV)], outs[1].scales)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_edge_4000x5000_full(dtype):
    """Without four-over-six; tests/test_gpu_fos_multitile.py has it with."""
    x = workloads.edge_normal(4000, 5000, dtype, DEV)
    for mode in (nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR):
        c = cfg(mode, 448.0)
        g, o = gpu_quantize(x, c), oracle_quantize(x, c)
        assert_same(g["row"], o["row"], f"row {mode}")
        assert_same(g["col"], o["col"], f"col {mode}")


@pytest.mark.parametrize("fos", [False, True])
def test_edge_8192_blocks_16x16_vs_1x16_sampled(fos):
    """8192 x 8192 per-tensor, 1x16 and 16x16 blocks, with and without four-over-six
    (4096 tiles: each CTA walks about 13), on strips of 16 rows in both layouts."""
    x = workloads.edge_normal(8192, 8192, torch.bfloat16, DEV, std=0.02)
    xb, tag = host_bits(x)
    _, _, t = oracle.amax(xb, tag)
    for b2d in (False, True):
        c = cfg(nv.NVFP4_PER_TENSOR, 448.0, fos, b2d)
        g = gpu_quantize(x, c)
        assert g["row"].amax.item() == t and g["col"].amax.item() == t
        for r0 in (0, 4096, 8176):
            strip = x[r0:r0 + 16]
            o = oracle_quantize(strip, c, row_amax_in=np.array([t], np.float32),
                                col_amax_in=np.array([t], np.float32))
            assert np.array_equal(g["row"].codes[r0:r0 + 16].cpu().numpy(), o["row"][0])
            assert np.array_equal(g["row"].scales[r0:r0 + 16].cpu().numpy(), o["row"][1])
            assert np.array_equal(g["col"].codes[:, r0 // 2:r0 // 2 + 8].cpu().numpy(),
                                  o["col"][0])
            assert np.array_equal(g["col"].scales[:, r0 // 16:r0 // 16 + 1].cpu().numpy(),
                                  o["col"][1])
        if b2d:
            # columnwise codes are the transpose of the rowwise codes
            rc, cc = g["row"].codes[:64, :32], g["col"].codes[:64, :32]
            rn = torch.stack([rc & 15, rc >> 4], -1).reshape(64, 64)
            cn = torch.stack([cc & 15, cc >> 4], -1).reshape(64, 64)
            assert torch.equal(rn, cn.t())


def test_edge_zero_rows_full():
    x = workloads.edge_zero_rows(device=DEV)
    c = cfg(nv.NVFP4_ROW_SCALED)
    g, o = gpu_quantize(x, c), oracle_quantize(x, c)
    assert_same(g["row"], o["row"]), assert_same(g["col"], o["col"])
    assert not g["row"].codes[::8].any()
