"""Grouped quantize from ragged tokens into the padded layout (GPU, through the C ABI).

The definition: the result equals zero-padding the ragged tokens into the padded
layout and quantizing that with per-group amax (nvfp4_grouped_quantize_rowwise,
NVFP4_PER_TENSOR), which the oracle computes on the padded tensor.  Checked byte
for byte against the oracle on small cases (empty groups, single rows, ragged tails,
FP32 and BF16, a width that no tensor map describes) and against the padded path
on the MoE workload; invalid layouts write nothing and set the status word.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads
from gpu_helpers import assert_same, cfg, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layout(counts, align=128):
    counts = np.asarray(counts, np.int64)
    padded = ((counts + align - 1) // align) * align
    return counts, padded, np.cumsum(counts), np.cumsum(padded)


def _ragged_and_padded(counts, cols, seed, dtype):
    counts, padded, rag_ends, pad_ends = _layout(counts)
    tokens, rows = int(counts.sum()), int(padded.sum())
    x = workloads.seeded_normal(max(tokens, 1), cols, seed=seed, dtype=dtype, device="cpu",
                                row_scale_decades=1.0)[:tokens]
    xp = torch.zeros(rows, cols, dtype=dtype)
    r0 = p0 = 0
    for c, p in zip(counts.tolist(), padded.tolist()):
        xp[p0:p0 + c] = x[r0:r0 + c]
        r0, p0 = r0 + c, p0 + p
    return x.contiguous(), xp, rag_ends, pad_ends


def _run_padded(x, rag_ends, pad_ends, rows, c, fill=None):
    cols = x.shape[1]
    out = nv.alloc_out(rows, cols, rows, DEV, fill)
    if fill is not None:
        out.amax.fill_(-1.0)
    ga = torch.full((len(rag_ends),), -1.0, device=DEV)
    nv.nvfp4_grouped_quantize_rowwise_padded(
        x.to(DEV), torch.from_numpy(np.asarray(rag_ends, np.int64)).to(DEV),
        torch.from_numpy(np.asarray(pad_ends, np.int64)).to(DEV), rows, c, out, ga)
    torch.cuda.synchronize()
    return out, ga


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fos,bound", [(True, 256.0), (False, 448.0)])
@pytest.mark.parametrize("cols", [256, 96, 100])
def test_padded_matches_oracle_on_padded_tensor(dtype, fos, bound, cols):
    x, xp, rag_ends, pad_ends = _ragged_and_padded([5, 0, 130, 128, 300, 1], cols, 21, dtype)
    rows = int(pad_ends[-1])
    c = cfg(nv.NVFP4_PER_TENSOR, bound, fos)
    out, ga = _run_padded(x, rag_ends, pad_ends, rows, c)
    xb, tag = host_bits(xp)
    codes, scales, ra, gam = oracle.grouped_quantize_rowwise(xb, tag, pad_ends, mode=0,
                                                              bound=bound, four_over_six=fos)
    assert_same(out, (codes, scales, ra), "padded")
    assert np.array_equal(ga.cpu().numpy(), gam)


def test_padded_equals_padded_path_on_moe_workload():
    xp, pad_ends, counts, padded = workloads.moe(DEV)
    x, rag_ends = workloads.moe_ragged(xp, counts, padded)
    rows, cols = xp.shape
    c = cfg(nv.NVFP4_PER_TENSOR, 256.0, True)
    ref = nv.alloc_out(rows, cols, rows, DEV)
    ga_ref = torch.empty(len(counts), device=DEV)
    nv.nvfp4_grouped_quantize_rowwise(xp, pad_ends, c, ref, ga_ref)
    out = nv.alloc_out(rows, cols, rows, DEV, 0xA5)
    ga = torch.empty(len(counts), device=DEV)
    nv.nvfp4_grouped_quantize_rowwise_padded(x.contiguous(), rag_ends.to(DEV), pad_ends, rows,
                                             c, out, ga)
    torch.cuda.synchronize()
    for name in ("codes", "scales", "amax"):
        assert torch.equal(getattr(out, name), getattr(ref, name)), name
    assert torch.equal(ga, ga_ref)


@pytest.mark.parametrize("case", ["short_padding", "misaligned_start", "bad_ragged_end"])
def test_invalid_layout_writes_nothing(case):
    counts = [130, 60]
    x, _, rag_ends, pad_ends = _ragged_and_padded(counts, 128, 22, torch.bfloat16)
    rag_ends, pad_ends = rag_ends.copy(), pad_ends.copy()
    if case == "short_padding":
        pad_ends[0] = 128  # group 0 has 130 tokens but only 128 padded rows
    elif case == "misaligned_start":
        pad_ends[:] = [136, 264]  # group 1 would start at row 136
    else:
        rag_ends[-1] = rag_ends[-1] - 1  # does not end at the token count
    rows = int(pad_ends[-1])
    nv.nvfp4_device_status(reset=True)
    out, ga = _run_padded(x, rag_ends, pad_ends, rows, cfg(nv.NVFP4_PER_TENSOR, 256.0, True),
                          fill=0xA5)
    assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS
    assert bool((out.codes == 0xA5).all()) and bool((out.scales == 0xA5).all())
    assert bool((ga == -1.0).all()) and bool((out.amax == -1.0).all())  # maxima untouched


def test_row_scaled_mode_is_unsupported():
    x, _, rag_ends, pad_ends = _ragged_and_padded([10], 64, 23, torch.bfloat16)
    with pytest.raises(nv.NVFP4Error):
        _run_padded(x, rag_ends, pad_ends, int(pad_ends[-1]),
                    cfg(nv.NVFP4_ROW_SCALED, 448.0, False))
