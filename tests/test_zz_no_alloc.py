"""nvfp4_gemm_static_ws: the GEMM with the library's static device workspace.

It must give exactly what nvfp4_gemm gives with a caller workspace (same kernels,
same arithmetic), on consecutive calls with different operands, allocate no device
memory, and reject a shape whose workspace does not fit before enqueueing anything.
"""
import numpy as np
import pytest
import torch

import nvfp4_precision_quantization_gb300 as nv
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
RS, PT = nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR


def _op(lines, k, seed, mode, bound=448.0):
    c, s, a = workloads.nvfp4_operand(lines, k, seed, row_scaled=mode == RS, device=DEV)
    return nv.Operand(c, s, a, mode, bound)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_static_workspace_matches_caller_workspace_on_two_calls(dtype):
    shapes = [(300, 520, 1024, RS, PT), (2048, 1024, 4096, RS, RS)]
    for i, (m, n, k, ma, mb) in enumerate(shapes):
        a, b = _op(m, k, 40 + 2 * i, ma), _op(n, k, 41 + 2 * i, mb, bound=256.0)
        ref = torch.full((m, n), float("nan"), dtype=dtype, device=DEV)
        got = torch.full((m, n), -1.0, dtype=dtype, device=DEV)
        nv.nvfp4_gemm(a, b, ref)
        nv.nvfp4_gemm_static_ws(a, b, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (m, n, k)
    assert nv.nvfp4_device_status(reset=True) == 0


def test_static_workspace_allocates_nothing():
    m, n, k = 1024, 2048, 2048
    a, b = _op(m, k, 50, RS), _op(n, k, 51, RS)
    d = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    nv.nvfp4_gemm_static_ws(a, b, d)  # first call on the device: kernels load
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        nv.nvfp4_gemm_static_ws(a, b, d)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_oversize_shape_is_rejected_and_writes_nothing():
    m, n, k = 65536, 8192, 16384  # needs 72 MiB of workspace
    assert nv.nvfp4_gemm_workspace_size(m, n, k) > nv.NVFP4_GEMM_STATIC_WS_BYTES
    # rejected on the host before any device access: the operand bytes are never read
    a = nv.Operand(torch.empty(m, k // 2, dtype=torch.uint8, device=DEV),
                   torch.empty(m, k // 16, dtype=torch.uint8, device=DEV),
                   torch.ones(m, device=DEV), RS, 448.0)
    b = nv.Operand(torch.empty(n, k // 2, dtype=torch.uint8, device=DEV),
                   torch.empty(n, k // 16, dtype=torch.uint8, device=DEV),
                   torch.ones(1, device=DEV), PT, 448.0)
    d = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nv.NVFP4Error) as ei:
        nv.nvfp4_gemm_static_ws(a, b, d)
    assert ei.value.status == nv.NVFP4_ERR_UNSUPPORTED
    assert "static workspace" in nv.nvfp4_last_error()
    torch.cuda.synchronize()
    assert bool((d == 3.0).all())
