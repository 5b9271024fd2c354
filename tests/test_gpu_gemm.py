"""NVFP4 GEMM consumer on the tensor cores (GPU, through the C ABI) against the
oracle's FP64 product of the dequantized operands.

Tolerance, from the arithmetic of the GPU path: every product of two block values
(code * decode(scale), E2M1 x E4M3) is exact in FP32, so the only errors are the
FP32 accumulation of k products in the tensor core's order (at most k * 2^-23 of
the sum of |terms|, allowing truncating partial sums), the two FP32 roundings of
each of alpha = amax_a * fl(1/F_a) and beta = amax_b * fl(1/F_b), fl(1/F) itself,
and the two multiplies of the epilogue (together under 8 * 2^-24 of the sum of
|terms|), then the output rounding: 2^-8 of |d| for BF16 (round to nearest even
is 2^-9; the slack covers the error already present) and 2^-23 for FP32.
    |d_gpu - d_exact| <= (k * 2^-23 + 2^-21) * sum|terms| + r_out * |d_exact|
The small cases keep k small enough (<= 1024, a bound of at most 2^-13 of the
magnitude) that a misplaced scale, row or K block -- an error of the size of a
whole term -- cannot hide inside it.

Operands are seeded synthetic NVFP4 bytes (workloads.nvfp4_operand) or the
oracle's own quantize of seeded data; nothing the oracle reads comes from the GPU.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
RS, PT = nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR


def _bound(k, dabs, dexact, bf16):
    return (k * 2.0 ** -23 + 2.0 ** -21) * dabs + (2.0 ** -8 if bf16 else 2.0 ** -23) * np.abs(dexact)


def _host_op(codes, scales, amax, mode, bound):
    return dict(codes=np.ascontiguousarray(codes), scales=np.ascontiguousarray(scales),
                amax=np.ascontiguousarray(amax, np.float32), row_scaled=mode == RS, bound=bound)


def _dev_op(h, mode):
    return nv.Operand(torch.from_numpy(h["codes"]).to(DEV), torch.from_numpy(h["scales"]).to(DEV),
                      torch.from_numpy(h["amax"]).to(DEV), mode, h["bound"])


def _random_op(lines, k, seed, mode, bound=448.0):
    c, s, a = workloads.nvfp4_operand(lines, k, seed, row_scaled=mode == RS)
    return _host_op(c.numpy(), s.numpy(), a.numpy(), mode, bound)


def _run(a_dev, b_dev, m, n, dtype):
    d = torch.full((m, n), float("nan"), dtype=dtype, device=DEV)
    nv.nvfp4_device_status(reset=True)
    nv.nvfp4_gemm(a_dev, b_dev, d)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status(reset=True) == 0
    return d.float().cpu().numpy().astype(np.float64)


def _compare(got, a_h, b_h, dtype, what):
    k = a_h["codes"].shape[1] * 2
    exp, dabs = oracle.gemm(a_h, b_h, with_abs=True)
    err = np.abs(got - exp)
    tol = _bound(k, dabs, exp, dtype == torch.bfloat16)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside the bound, first "
                           f"{bad[:4].tolist()}: got {got[tuple(bad[0])]} want {exp[tuple(bad[0])]}")


SHAPES = [(128, 256, 256), (1, 1, 32), (200, 300, 512), (64, 96, 96), (129, 257, 288),
          (256, 512, 1024)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("modes", [(RS, RS), (RS, PT), (PT, RS), (PT, PT)])
def test_gemm_matches_oracle(shape, modes):
    m, n, k = shape
    a_h = _random_op(m, k, 1, modes[0])
    b_h = _random_op(n, k, 2, modes[1], bound=256.0)
    dtype = torch.bfloat16 if (m + n) % 2 == 0 else torch.float32
    got = _run(_dev_op(a_h, modes[0]), _dev_op(b_h, modes[1]), m, n, dtype)
    _compare(got, a_h, b_h, dtype, f"{shape} {modes}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gemm_output_dtypes_on_tile_edges(dtype):
    m, n, k = 257, 255, 544  # ragged in every dimension; k not a multiple of 64
    a_h = _random_op(m, k, 3, RS)
    b_h = _random_op(n, k, 4, RS)
    _compare(_run(_dev_op(a_h, RS), _dev_op(b_h, RS), m, n, dtype), a_h, b_h, dtype, "edges")


def test_fprop_and_wgrad_on_quantized_operands():
    """The two GEMMs of the row-scaled linear layer: fprop Y = X W^T with X row-scaled
    rowwise and W per-tensor; wgrad dW = dY^T X with both columnwise and row-scaled
    (per-column amax), the bilateral case.  Operands are the oracle's quantize."""
    rng = np.random.default_rng(11)
    tokens, d_in, d_out = 256, 192, 320
    x = (rng.standard_normal((tokens, d_in)) * np.exp(rng.uniform(-2, 2, (tokens, 1)))).astype(np.float32)
    w = (rng.standard_normal((d_out, d_in)) * 0.05).astype(np.float32)
    dy = (rng.standard_normal((tokens, d_out)) * np.exp(rng.uniform(-2, 2, (tokens, 1)))).astype(np.float32)
    qx = oracle.quantize(x, "fp32", mode=oracle.ROW_SCALED)
    qw = oracle.quantize(w, "fp32", mode=oracle.PER_TENSOR, bound=256.0, four_over_six=True,
                         columnwise=False)
    qdy = oracle.quantize(dy, "fp32", mode=oracle.ROW_SCALED, rowwise=False)
    # fprop: A = X rowwise (per-row amax), B = W rowwise (per-tensor amax)
    a_h = _host_op(*qx["row"], RS, 448.0)
    b_h = _host_op(*qw["row"], PT, 256.0)
    y = _run(_dev_op(a_h, RS), _dev_op(b_h, PT), tokens, d_out, torch.bfloat16)
    _compare(y, a_h, b_h, torch.bfloat16, "fprop")
    # the result approximates the unquantized product
    ref = x.astype(np.float64) @ w.T.astype(np.float64)
    assert np.linalg.norm(y - ref) < 0.2 * np.linalg.norm(ref)
    # wgrad: A = dY columnwise (lines = output features), B = X columnwise (input features)
    a_h = _host_op(*qdy["col"], RS, 448.0)
    b_h = _host_op(*qx["col"], RS, 448.0)
    dw = _run(_dev_op(a_h, RS), _dev_op(b_h, RS), d_out, d_in, torch.float32)
    _compare(dw, a_h, b_h, torch.float32, "wgrad")
    ref = dy.T.astype(np.float64) @ x.astype(np.float64)
    assert np.linalg.norm(dw - ref) < 0.2 * np.linalg.norm(ref)


@pytest.mark.parametrize("which", ["fprop", "wgrad"])
def test_full_size_linear_gemm_sampled(which):
    """The bench's GEMM shapes, full size, in its launch configuration; 48 x 48
    outputs (tile corners and random positions) against the oracle."""
    m, n, k = workloads.GEMM_SHAPES[which]
    ca, sa, aa = workloads.nvfp4_operand(m, k, 21, row_scaled=True, device=DEV)
    cb, sb, ab = workloads.nvfp4_operand(n, k, 22, row_scaled=which == "wgrad", device=DEV)
    mb = RS if which == "wgrad" else PT
    d = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    nv.nvfp4_device_status(reset=True)
    nv.nvfp4_gemm(nv.Operand(ca, sa, aa, RS, 448.0), nv.Operand(cb, sb, ab, mb, 448.0), d)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status(reset=True) == 0
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, m - 1], rng.integers(0, m, 44)]))
    cols = np.unique(np.concatenate([[0, 255, 256, n - 1], rng.integers(0, n, 44)]))
    ri, ci = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    a_h = _host_op(ca[ri].cpu().numpy(), sa[ri].cpu().numpy(), aa[ri].cpu().numpy(), RS, 448.0)
    bam = ab[ci] if mb == RS else ab
    b_h = _host_op(cb[ci].cpu().numpy(), sb[ci].cpu().numpy(), bam.cpu().numpy(), mb, 448.0)
    got = d[ri][:, ci].float().cpu().numpy().astype(np.float64)
    _compare(got, a_h, b_h, torch.bfloat16, which)


def test_empty_k_writes_zeros_and_empty_mn_writes_nothing():
    a = _dev_op(_random_op(8, 32, 6, RS), RS)
    b = _dev_op(_random_op(8, 32, 7, RS), RS)
    a0 = nv.Operand(a.codes[:, :0], a.scales[:, :0], a.amax, RS, 448.0)
    b0 = nv.Operand(b.codes[:, :0], b.scales[:, :0], b.amax, RS, 448.0)
    d = torch.full((8, 8), 7.0, device=DEV)
    nv.nvfp4_gemm(a0, b0, d)
    torch.cuda.synchronize()
    assert bool((d == 0).all())
    e = torch.full((0, 8), 7.0, device=DEV)
    nv.nvfp4_gemm(nv.Operand(a.codes[:0], a.scales[:0], a.amax, RS, 448.0), b, e)
    torch.cuda.synchronize()


def test_k_not_multiple_of_32_is_unsupported():
    a = _dev_op(_random_op(4, 48, 8, RS), RS)
    d = torch.empty(4, 4, device=DEV)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.nvfp4_gemm(a, a, d)
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED


def test_repeated_calls_agree_and_overwrite():
    """Same inputs, two calls on one workspace: identical outputs (the result does not
    depend on what the output or workspace held before)."""
    m, n, k = 300, 600, 2048
    a = _dev_op(_random_op(m, k, 9, RS), RS)
    b = _dev_op(_random_op(n, k, 10, PT), PT)
    ws = torch.full((nv.nvfp4_gemm_workspace_size(m, n, k),), 0xFF, dtype=torch.uint8, device=DEV)
    d1 = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    d2 = torch.full((m, n), -5.0, dtype=torch.bfloat16, device=DEV)
    nv.nvfp4_gemm(a, b, d1, ws)
    nv.nvfp4_gemm(a, b, d2, ws)
    torch.cuda.synchronize()
    assert torch.equal(d1, d2)


@pytest.mark.parametrize("shape", [(256, 512, 1024), (129, 300, 544)])
def test_accumulation_is_exact_on_representable_operands(shape):
    """Operands whose every partial sum is exactly representable in FP32: code
    magnitudes in {0, .5, ..., 6} (multiples of 0.5, at most 6) times power-of-two
    scales 0.5 .. 4, amax = F (value = code * scale): each product is a multiple of
    2^-4 below 2^10, and any partial sum of at most 1024 of them is below 2^20 -- 24
    significant bits -- so the tensor core's FP32 accumulation is exact in any order.
    Then d = fl(fl(acc * alpha) * beta) with acc the exact product, alpha = fl(F *
    fl(1/F)), beta likewise: the GPU must match that bit for bit."""
    m, n, k = shape
    rng = np.random.default_rng(17)
    F = 448.0 * 6.0

    def op(lines):
        codes = rng.integers(0, 256, (lines, k // 2), dtype=np.uint8)
        scales = rng.choice(np.array([0x30, 0x38, 0x40, 0x48], np.uint8), (lines, k // 16))
        return _host_op(codes, scales, np.full(lines, F, np.float32), RS, 448.0)

    a_h, b_h = op(m), op(n)
    got = _run(_dev_op(a_h, RS), _dev_op(b_h, RS), m, n, torch.float32)
    exact = oracle.gemm(a_h, b_h)  # amax / F = 1: the plain sum of code * scale products
    assert np.all(np.abs(exact) < 2.0 ** 20) and np.all(exact * 16 == np.round(exact * 16))
    f32 = np.float32
    alpha = f32(f32(F) * (f32(1.0) / f32(F)))
    want = (exact.astype(f32) * alpha).astype(f32) * alpha
    assert np.array_equal(got.astype(f32).view(np.uint32), want.astype(f32).view(np.uint32))


def test_fprop_with_16x16_block_weight():
    """A 16x16-block weight (per-tensor, "Add backward overrides and 1x16 weights to
    NVFP4 four-over-six", torchao PR #8) is a valid B operand as the quantize entry
    points write it: its rowwise scales carry each tile's scale on all 16 lines."""
    rng = np.random.default_rng(12)
    tokens, d_in, d_out = 200, 256, 272
    x = (rng.standard_normal((tokens, d_in)) * np.exp(rng.uniform(-2, 2, (tokens, 1)))).astype(np.float32)
    w = (rng.standard_normal((d_out, d_in)) * 0.05).astype(np.float32)
    qx = oracle.quantize(x, "fp32", mode=oracle.ROW_SCALED, columnwise=False)
    qw = oracle.quantize(w, "fp32", mode=oracle.PER_TENSOR, block_2d=True, columnwise=False)
    sw = qw["row"][1]
    assert np.array_equal(sw[0::16], sw[15::16])  # the tile's scale on each of its lines
    a_h = _host_op(*qx["row"], RS, 448.0)
    b_h = _host_op(*qw["row"], PT, 448.0)
    y = _run(_dev_op(a_h, RS), _dev_op(b_h, PT), tokens, d_out, torch.bfloat16)
    _compare(y, a_h, b_h, torch.bfloat16, "fprop 16x16 weight")
