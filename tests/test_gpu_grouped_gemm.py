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


# ---------------------------------------------------------------- wgrad (K grouped)

def _wgrad_run(a_h, b_h, ends, a_mode, b_mode, dtype, fill=float("nan")):
    G, m, n = len(ends), a_h["codes"].shape[0], b_h["codes"].shape[0]
    d = torch.full((G, m, n), fill, dtype=dtype, device=DEV)
    nv.nvfp4_device_status(reset=True)
    nv.nvfp4_grouped_gemm_wgrad(_dev(a_h, a_mode), _dev(b_h, b_mode),
                                torch.tensor(ends, dtype=torch.int64, device=DEV), d)
    torch.cuda.synchronize()
    return d


@pytest.mark.parametrize("modes", [(RS, RS), (PT, PT), (RS, PT)])
def test_grouped_wgrad_matches_oracle(modes):
    ends = [256, 256, 768, 1024]  # an empty group
    G, m, n, tokens = len(ends), 200, 300, ends[-1]
    ca, sa, _ = workloads.nvfp4_operand(m, tokens, 80, row_scaled=True)
    cb, sb, _ = workloads.nvfp4_operand(n, tokens, 81, row_scaled=True)
    rng = np.random.default_rng(9)
    aa = np.exp(rng.uniform(-2, 2, G * m if modes[0] == RS else G)).astype(np.float32)
    ab = np.exp(rng.uniform(-2, 2, G * n if modes[1] == RS else G)).astype(np.float32)
    a_h = _host_op(ca.numpy(), sa.numpy(), aa, modes[0], 448.0)
    b_h = _host_op(cb.numpy(), sb.numpy(), ab, modes[1], 256.0)
    dtype = torch.float32 if modes[0] == modes[1] else torch.bfloat16
    d = _wgrad_run(a_h, b_h, ends, modes[0], modes[1], dtype)
    assert nv.nvfp4_device_status(reset=True) == 0
    got = d.float().cpu().numpy().astype(np.float64)
    exp, dabs = oracle.grouped_gemm_wgrad(a_h, b_h, ends, with_abs=True)
    assert np.all(got[1] == 0)  # the empty group
    bad = np.argwhere(~(np.abs(got - exp) <= _bound(512, dabs, exp, dtype == torch.bfloat16)))
    assert bad.size == 0, f"{len(bad)} outside the bound, first {bad[:4].tolist()}"


def test_grouped_wgrad_on_grouped_columnwise_operands():
    """The MoE backward chain: dY and X of two token groups quantized columnwise per
    group (row-scaled: each group's column amax; the oracle's quantize, group by group),
    then dW_g = dY_g^T X_g on the tensor cores against the oracle."""
    rng = np.random.default_rng(10)
    ends = [256, 768]
    d_out, d_in, tokens = 256, 192, ends[-1]
    dy = (rng.standard_normal((tokens, d_out)) * 0.5).astype(np.float32)
    x = (rng.standard_normal((tokens, d_in)) * np.exp(rng.uniform(-1, 1, (tokens, 1)))).astype(np.float32)

    def per_group_columnwise(t):
        cols = t.shape[1]
        codes = np.zeros((cols, tokens // 2), np.uint8)
        scales = np.zeros((cols, tokens // 16), np.uint8)
        amax = np.zeros((len(ends), cols), np.float32)
        s = 0
        for g, e in enumerate(ends):
            o = oracle.quantize(t[s:e], "fp32", mode=oracle.ROW_SCALED, rowwise=False)["col"]
            codes[:, s // 2:e // 2], scales[:, s // 16:e // 16], amax[g] = o
            s = e
        return _host_op(codes, scales, amax.reshape(-1), RS, 448.0)

    a_h, b_h = per_group_columnwise(dy), per_group_columnwise(x)
    d = _wgrad_run(a_h, b_h, ends, RS, RS, torch.float32)
    assert nv.nvfp4_device_status(reset=True) == 0
    got = d.cpu().numpy().astype(np.float64)
    exp, dabs = oracle.grouped_gemm_wgrad(a_h, b_h, ends, with_abs=True)
    assert np.all(np.abs(got - exp) <= _bound(512, dabs, exp, False))
    s = 0
    for g, e in enumerate(ends):  # close to the unquantized per-group product
        ref = dy[s:e].T.astype(np.float64) @ x[s:e].astype(np.float64)
        assert np.linalg.norm(got[g] - ref) < 0.2 * np.linalg.norm(ref), g
        s = e


def test_grouped_wgrad_invalid_ends_write_nothing():
    m = n = 128
    tokens = 512
    ca, sa, _ = workloads.nvfp4_operand(m, tokens, 90, row_scaled=True)
    cb, sb, _ = workloads.nvfp4_operand(n, tokens, 91, row_scaled=True)
    for ends in ([128, 512], [512, 256], [256]):  # unaligned, decreasing, short
        G = len(ends)
        a_h = _host_op(ca.numpy(), sa.numpy(), np.ones(G * m, np.float32), RS, 448.0)
        b_h = _host_op(cb.numpy(), sb.numpy(), np.ones(G * n, np.float32), RS, 448.0)
        d = _wgrad_run(a_h, b_h, ends, RS, RS, torch.float32, fill=7.0)
        assert nv.nvfp4_device_status(reset=True) & nv.NVFP4_DEVICE_BAD_GROUPS, ends
        assert bool((d == 7.0).all()), ends


def test_grouped_wgrad_tokens_not_multiple_of_256_is_unsupported():
    ca, sa, _ = workloads.nvfp4_operand(128, 384, 92, row_scaled=True)
    a_h = _host_op(ca.numpy(), sa.numpy(), np.ones(128, np.float32), RS, 448.0)
    with pytest.raises(nv.NVFP4Error) as ei:
        _wgrad_run(a_h, a_h, [384], RS, RS, torch.float32)
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED


def test_more_groups_than_staged_in_shared_memory():
    """600 groups (more than the kernel stages in shared memory, so every tile looks
    its group up in global memory), nearly all empty, in both grouped modes."""
    n, k = 256, 64
    ends = [0] * 299 + [128] * 299 + [384, 512]
    a_h, b_h = _operands(ends[-1], len(ends), n, k, 100, RS)
    d = _run(a_h, b_h, ends, n, torch.float32, RS)
    assert nv.nvfp4_device_status(reset=True) == 0
    exp, dabs = oracle.grouped_gemm(a_h, b_h, ends, n, with_abs=True)
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - exp) <= _bound(k, dabs, exp, False))

    ends = [0] * 300 + [256] * 200 + [768] * 99 + [1024]
    G, m, n, tokens = len(ends), 128, 256, ends[-1]
    ca, sa, _ = workloads.nvfp4_operand(m, tokens, 102, row_scaled=True)
    cb, sb, _ = workloads.nvfp4_operand(n, tokens, 103, row_scaled=True)
    rng = np.random.default_rng(12)
    a_h = _host_op(ca.numpy(), sa.numpy(), np.exp(rng.uniform(-2, 2, G * m)).astype(np.float32),
                   RS, 448.0)
    b_h = _host_op(cb.numpy(), sb.numpy(), np.exp(rng.uniform(-2, 2, G * n)).astype(np.float32),
                   RS, 448.0)
    d = _wgrad_run(a_h, b_h, ends, RS, RS, torch.float32)
    assert nv.nvfp4_device_status(reset=True) == 0
    got = d.cpu().numpy().astype(np.float64)
    exp, dabs = oracle.grouped_gemm_wgrad(a_h, b_h, ends, with_abs=True)
    assert np.all(got[:300] == 0) and np.all(got[301:500] == 0) and np.all(got[501:599] == 0)
    assert np.all(np.abs(got - exp) <= _bound(512, dabs, exp, False))
