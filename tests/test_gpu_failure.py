"""The failure path of the bounded waits, made to run on the GPU without a fault.

Every mbarrier wait in the pipeline kernels is bounded; a wait that gives up sets
NVFP4_DEVICE_TIMEOUT in the library's status word and the kernel returns without
writing its outputs.  nvfp4_selftest_wait_timeout runs that same wait on an
mbarrier that nothing ever arrives on, with a limit of a few milliseconds, so the
wait always runs out; nothing else is in flight when it does.
"""
import ctypes
import time

import pytest
import torch

from tests.gpu_helpers import assert_same, cfg, gpu_quantize, oracle_quantize
import workloads

nv = pytest.importorskip("nvfp4_precision_quantization_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_bounded_wait_gives_up_sets_status_and_writes_nothing():
    nv.nvfp4_device_status(reset=True)
    out = torch.full((1,), 7, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    nv.nvfp4_selftest_wait_timeout(2_000_000, out)  # 2 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert out.item() == 7  # the wait did not complete, so nothing was written
    assert elapsed < 1.0
    assert nv.nvfp4_device_status() & nv.NVFP4_DEVICE_TIMEOUT
    # through the C ABI: the status call reports NVFP4_ERR_TIMEOUT with a message
    v = ctypes.c_int32(0)
    rc = nv.load_library().nvfp4_device_status(ctypes.byref(v), 1)
    assert rc == nv.NVFP4_ERR_TIMEOUT and v.value & nv.NVFP4_DEVICE_TIMEOUT
    assert "bounded wait" in nv.nvfp4_last_error()
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_selftest_wait_timeout(1_000_000, out)
        nv.nvfp4_device_status(reset=True, raise_on_timeout=True)
    assert nv.nvfp4_device_status() == 0


def test_context_usable_after_a_timeout():
    nv.nvfp4_device_status(reset=True)
    out = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(3):
        nv.nvfp4_selftest_wait_timeout(500_000, out)
    assert nv.nvfp4_device_status(reset=True) == nv.NVFP4_DEVICE_TIMEOUT
    x = workloads.tiny(DEV)
    c = cfg(nv.NVFP4_ROW_SCALED, 448.0)
    g, o = gpu_quantize(x, c), oracle_quantize(x, c)
    assert_same(g["row"], o["row"], "row")
    assert_same(g["col"], o["col"], "col")
    assert nv.nvfp4_device_status() == 0
    assert out.item() == 0
