"""Grouped (per-expert) NVFP4 GEMM on the tensor cores (GPU, through the C ABI)
against the oracle's per-group FP64 product, within the bound derived for the GEMM
(tests/test_gpu_gemm.py): group g's token rows times expert g's weight rows, with
the bilateral amax post-scale ("Add NVFP4 four-over-six grouped GEMM for MoE
training", torchao PR #9, description)."""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads
from test_gpu_gemm import _bound, _host_op

pytestmark = pytest.mark.gpu
DEV = "cuda"
RS, PT = nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR


def _dev(h, mode):
    return nv.Operand(torch.from_numpy(h["codes"]).to(DEV), torch.from_numpy(h["scales"]).to(DEV),
                      torch.from_numpy(h["amax"]).to(DEV), mode, h["bound"])


def _operands(rows, groups, n, k, seed, b_mode):
    ca, sa, aa = workloads.nvfp4_operand(rows, k, seed, row_scaled=True)
    cb, sb, ab = workloads.nvfp4_operand(groups * n, k, seed + 1, row_scaled=True)
    if b_mode == PT:
        ab = ab[:groups].clone()  # one amax per expert
    return (_host_op(ca.numpy(), sa.numpy(), aa.numpy(), RS, 448.0),
            _host_op(cb.numpy(), sb.numpy(), ab.numpy(), b_mode, 256.0))


def _run(a_h, b_h, ends, n, dtype, b_mode, fill=float("nan")):
    rows = a_h["codes"].shape[0]
    d = torch.full((rows, n), fill, dtype=dtype, device=DEV)
    nv.nvfp4_device_status(reset=True)
    nv.nvfp4_grouped_gemm(_dev(a_h, RS), _dev(b_h, b_mode),
                          torch.tensor(ends, dtype=torch.int64, device=DEV), d)
    torch.cuda.synchronize()
    return d


@pytest.mark.parametrize("b_mode", [RS, PT])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_grouped_gemm_matches_oracle(b_mode, dtype):
    ends = [128, 128, 384, 512, 512]  # empty groups first-but-one and last
    n, k = 512, 544
    a_h, b_h = _operands(ends[-1], len(ends), n, k, 40, b_mode)
    d = _run(a_h, b_h, ends, n, dtype, b_mode)
    assert nv.nvfp4_device_status(reset=True) == 0
    got = d.float().cpu().numpy().astype(np.float64)
    exp, dabs = oracle.grouped_gemm(a_h, b_h, ends, n, with_abs=True)
    bad = np.argwhere(~(np.abs(got - exp) <= _bound(k, dabs, exp, dtype == torch.bfloat16)))
    assert bad.size == 0, f"{len(bad)} outside the bound, first {bad[:4].tolist()}"


def test_invalid_group_ends_write_nothing():
    n, k = 256, 256
    a_h, b_h = _operands(256, 2, n, k, 50, RS)
    for ends in ([100, 256], [256, 128], [128, 200]):  # unaligned, decreasing, short
        d = _run(a_h, b_h, ends, n, torch.float32, RS, fill=7.0)
        assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS, ends
        assert bool((d == 7.0).all()), ends


def test_n_not_multiple_of_256_is_unsupported():
    a_h, b_h = _operands(128, 1, 192, 64, 60, RS)
    with pytest.raises(nv.NVFP4Error) as ei:
        _run(a_h, b_h, [128], 192, torch.float32, RS)
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED


def test_moe_grouped_gemm_sampled():
    """The MoE bench shape: the padded tokens of the 32-group workload (K 7168) times
    32 experts of N 2048, per-expert weight amax; 40 rows per sampled group against
    the oracle."""
    _, _, pad_ends = workloads.moe_layout()
    ends = pad_ends.numpy()
    rows, n, k, G = int(ends[-1]), 2048, 7168, len(ends)
    ca, sa, aa = workloads.nvfp4_operand(rows, k, 70, row_scaled=True, device=DEV)
    cb, sb, ab = workloads.nvfp4_operand(G * n, k, 71, row_scaled=False, device=DEV)
    ab = torch.rand(G, device=DEV) + 0.5
    d = torch.empty(rows, n, dtype=torch.bfloat16, device=DEV)
    nv.nvfp4_device_status(reset=True)
    nv.nvfp4_grouped_gemm(nv.Operand(ca, sa, aa, RS, 448.0), nv.Operand(cb, sb, ab, PT, 448.0),
                          pad_ends.to(DEV), d)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status(reset=True) == 0
    rng = np.random.default_rng(8)
    cols = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 30)]))
    ci = torch.from_numpy(cols).to(DEV)
    for g in (0, G // 2, G - 1):
        s = int(ends[g - 1]) if g else 0
        e = int(ends[g])
        if e == s:
            continue
        r = np.unique(np.concatenate([[s, e - 1], rng.integers(s, e, 38)]))
        ri = torch.from_numpy(r).to(DEV)
        a_h = _host_op(ca[ri].cpu().numpy(), sa[ri].cpu().numpy(), aa[ri].cpu().numpy(), RS, 448.0)
        bi = ci + g * n
        b_h = _host_op(cb[bi].cpu().numpy(), sb[bi].cpu().numpy(), ab[g:g + 1].cpu().numpy(), PT,
                       448.0)
        exp, dabs = oracle.gemm(a_h, b_h, with_abs=True)
        got = d[ri][:, ci].float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - exp) <= _bound(k, dabs, exp, True)), g
