"""Grouped columnwise quantize (GPU, through the C ABI).

Definition: each group's rows are quantized columnwise on their own (row-scaled:
a column's amax over the group's rows; per-tensor: the group's amax) and the results
sit side by side along the token axis of the columnwise layout.  The oracle computes
exactly that, group by group, and the GPU output must match byte for byte.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads
from gpu_helpers import cfg, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _expected(x, ends, c, mask=None):
    """Oracle, one group at a time, concatenated along the token axis (mask: of the
    transform of x instead of x)."""
    xb, tag = host_bits(x)
    if mask is not None:
        xb, tag = oracle.rht16(xb, tag, mask), "fp32"
    rows, cols = xb.shape
    codes = np.zeros((cols, rows // 2), np.uint8)
    scales = np.zeros((cols, rows // 16), np.uint8)
    rs = c.mode == nv.NVFP4_ROW_SCALED
    amax = np.zeros((len(ends), cols) if rs else (len(ends),), np.float32)
    start = 0
    for g, e in enumerate(np.asarray(ends).tolist()):
        if e > start:
            o = oracle.quantize(xb[start:e], tag, mode=c.mode, bound=c.bound,
                                four_over_six=bool(c.four_over_six), rowwise=False)["col"]
            codes[:, start // 2:e // 2] = o[0]
            scales[:, start // 16:e // 16] = o[1]
            amax[g] = o[2] if rs else o[2][0]
        start = e
    return codes, scales, amax


def _run(x, ends, c, amax_in=None, fill=None, mask=None, noop=None):
    rows, cols = x.shape
    G = len(ends)
    rs = c.mode == nv.NVFP4_ROW_SCALED
    col = nv.alloc_out(cols, rows, G * cols if rs else G, DEV, fill)
    if fill is not None:
        col.amax.fill_(-1.0)
    col.amax_in = amax_in
    e = torch.from_numpy(np.asarray(ends, np.int64)).to(DEV)
    if mask is None:
        nv.nvfp4_grouped_quantize_columnwise(x, e, c, col, noop=noop)
    else:
        nv.nvfp4_grouped_quantize_columnwise_rht(x, e, mask, c, col, noop=noop)
    torch.cuda.synchronize()
    return col


def _check(col, exp, what):
    codes, scales, amax = exp
    got = col.codes.cpu().numpy(), col.scales.cpu().numpy(), col.amax.cpu().numpy()
    assert np.array_equal(got[0], codes), f"{what}: codes differ at {np.argwhere(got[0] != codes)[:5]}"
    assert np.array_equal(got[1], scales), f"{what}: scales differ"
    assert np.array_equal(got[2].reshape(amax.shape).view(np.uint32), amax.view(np.uint32)), what


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("fos,bound", [(False, 448.0), (True, 256.0)])
@pytest.mark.parametrize("cols", [256, 200, 96])
def test_grouped_columnwise_matches_oracle(dtype, mode, fos, bound, cols):
    ends = np.cumsum([128, 0, 256, 384, 128])
    x = workloads.seeded_normal(int(ends[-1]), cols, seed=31, dtype=dtype, device=DEV,
                                row_scale_decades=1.0)
    c = cfg(mode, bound, fos)
    _check(_run(x, ends, c), _expected(x, ends, c), "grouped columnwise")


def test_given_amax_gives_the_same_result():
    ends = np.cumsum([256, 128])
    x = workloads.seeded_normal(int(ends[-1]), 192, seed=32, device=DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    ref = _run(x, ends, c)
    given = ref.amax.clone()
    col = _run(x, ends, c, amax_in=given)
    assert torch.equal(col.codes, ref.codes) and torch.equal(col.scales, ref.scales)
    assert torch.equal(col.amax, ref.amax)


def test_moe_workload_groups_match_oracle():
    xp, ends, counts, padded = workloads.moe(DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    ends_np = ends.cpu().numpy()
    col = _run(xp, ends_np, c)
    # two groups in full against the oracle (the whole tensor is ~1 GB)
    for g in (0, len(ends_np) - 1):
        s, e = (int(ends_np[g - 1]) if g else 0), int(ends_np[g])
        xb, tag = host_bits(xp[s:e])
        o = oracle.quantize(xb, tag, mode=c.mode, bound=c.bound, rowwise=False)["col"]
        assert np.array_equal(col.codes[:, s // 2:e // 2].cpu().numpy(), o[0]), g
        assert np.array_equal(col.scales[:, s // 16:e // 16].cpu().numpy(), o[1]), g
        assert np.array_equal(col.amax.view(len(ends_np), -1)[g].cpu().numpy(), o[2]), g


def test_unaligned_ends_write_nothing():
    ends = np.array([100, 256], np.int64)  # group 0 ends inside a 128-row tile
    x = workloads.seeded_normal(256, 128, seed=33, device=DEV)
    nv.nvfp4_device_status(reset=True)
    col = _run(x, ends, cfg(nv.NVFP4_ROW_SCALED, 448.0, False), fill=0xA5)
    assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS
    assert bool((col.codes == 0xA5).all()) and bool((col.scales == 0xA5).all())
    assert bool((col.amax == -1.0).all())


# ---------------------------------------------------------------- with the transform

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("fos,bound", [(False, 448.0), (True, 256.0)])
@pytest.mark.parametrize("cols", [256, 96])
def test_grouped_columnwise_rht_matches_oracle(dtype, mode, fos, bound, cols):
    """Each group's rows transformed block by block (16 tokens per block, groups of
    whole 128-row tiles) and quantized with the group's amax of the transform."""
    ends = np.cumsum([128, 0, 256, 384, 128])
    x = workloads.seeded_normal(int(ends[-1]), cols, seed=34, dtype=dtype, device=DEV,
                                row_scale_decades=1.0)
    c = cfg(mode, bound, fos)
    _check(_run(x, ends, c, mask=0xC3A5), _expected(x, ends, c, mask=0xC3A5),
           "grouped columnwise rht")


def test_grouped_columnwise_rht_equals_transform_then_quantize():
    """The fused call gives the bytes of the transform into a buffer followed by the
    plain grouped columnwise quantize of that buffer, on the MoE tokens."""
    xp, ends, _, _ = workloads.moe(DEV)
    xp = xp[:int(ends[7])]  # the first 8 groups
    e = ends[:8].contiguous()
    for c in (cfg(nv.NVFP4_ROW_SCALED, 448.0, False), cfg(nv.NVFP4_PER_TENSOR, 256.0, True)):
        fused = _run(xp, e.cpu().numpy(), c, mask=0x6D2B)
        y = torch.empty(xp.shape, dtype=torch.float32, device=DEV)
        nv.nvfp4_rht16(xp, 0x6D2B, y)
        two = _run(y, e.cpu().numpy(), c)
        assert torch.equal(fused.codes, two.codes) and torch.equal(fused.scales, two.scales)
        assert torch.equal(fused.amax, two.amax)


def test_grouped_columnwise_rht_moe_groups_match_oracle():
    xp, ends, _, _ = workloads.moe(DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0, False)
    ends_np = ends.cpu().numpy()
    col = _run(xp, ends_np, c, mask=0x6D2B)
    for g in (0, len(ends_np) - 1):
        s, e = (int(ends_np[g - 1]) if g else 0), int(ends_np[g])
        xb, tag = host_bits(xp[s:e])
        o = oracle.quantize_columnwise_rht(xb, tag, 0x6D2B, mode=c.mode, bound=c.bound)
        assert np.array_equal(col.codes[:, s // 2:e // 2].cpu().numpy(), o[0]), g
        assert np.array_equal(col.scales[:, s // 16:e // 16].cpu().numpy(), o[1]), g
        assert np.array_equal(col.amax.view(len(ends_np), -1)[g].cpu().numpy(), o[2]), g


def test_grouped_columnwise_rht_unaligned_ends_and_noop_write_nothing():
    x = workloads.seeded_normal(256, 128, seed=35, device=DEV)
    nv.nvfp4_device_status(reset=True)
    col = _run(x, np.array([100, 256], np.int64), cfg(nv.NVFP4_ROW_SCALED, 448.0, False),
               fill=0xA5, mask=0x1)
    assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS
    assert bool((col.codes == 0xA5).all()) and bool((col.scales == 0xA5).all())
    assert bool((col.amax == -1.0).all())
    noop = torch.ones(1, dtype=torch.float32, device=DEV)
    col = _run(x, np.array([128, 256], np.int64), cfg(nv.NVFP4_PER_TENSOR, 448.0, False),
               fill=0xA5, mask=0x1, noop=noop)
    assert bool((col.codes == 0xA5).all()) and bool((col.amax == -1.0).all())
