"""The C-ABI library builds, loads, and exports every entry point that
include/nvfp4.h declares (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from nvfp4_precision_quantization_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("nvfp4_amax", "nvfp4_quantize_rowwise", "nvfp4_quantize_columnwise",
                 "nvfp4_quantize_both", "nvfp4_dequantize", "nvfp4_grouped_amax",
                 "nvfp4_grouped_quantize_rowwise", "nvfp4_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib_path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {n for n in exported if n.startswith("nvfp4_")}
    assert ours == set(declared_functions())


def test_binding_wraps_every_symbol(lib_path):
    import nvfp4_precision_quantization_gb300 as nv
    assert set(nv.EXPORTED_SYMBOLS) == set(declared_functions())
    nv.load_library()
    for name in declared_functions():
        assert callable(getattr(nv, name))


def test_host_validation_without_gpu(lib_path):
    """Argument checks run before any CUDA call, so they work on a CPU host."""
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 300.0, 0, 0)  # bad bound
    out = nv._COut(1, 1, 1, None)
    st = L.nvfp4_quantize_rowwise(16, nv.NVFP4_IN_BF16, 4, 4, ctypes.byref(cfg),
                                  ctypes.byref(out), None, None)
    assert st == nv.NVFP4_ERR_INVALID and "bound" in nv.nvfp4_last_error()
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 1)  # 16x16 with row-scaled
    st = L.nvfp4_quantize_rowwise(16, nv.NVFP4_IN_BF16, 4, 4, ctypes.byref(cfg),
                                  ctypes.byref(out), None, None)
    assert st == nv.NVFP4_ERR_INVALID and "16x16" in nv.nvfp4_last_error()
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
    st = L.nvfp4_quantize_rowwise(16, 7, 4, 4, ctypes.byref(cfg), ctypes.byref(out), None, None)
    assert st == nv.NVFP4_ERR_INVALID and "dtype" in nv.nvfp4_last_error()
    st = L.nvfp4_quantize_rowwise(16, nv.NVFP4_IN_BF16, -1, 4, ctypes.byref(cfg),
                                  ctypes.byref(out), None, None)
    assert st == nv.NVFP4_ERR_INVALID
    st = L.nvfp4_quantize_rowwise(None, nv.NVFP4_IN_BF16, 4, 4, ctypes.byref(cfg),
                                  ctypes.byref(out), None, None)
    assert st == nv.NVFP4_ERR_INVALID and "x is NULL" in nv.nvfp4_last_error()
    st = L.nvfp4_dequantize(1, 1, 1, nv.NVFP4_ROW_SCALED, 4, 4, 448.0, 1, 9, None)
    assert st == nv.NVFP4_ERR_INVALID
    st = L.nvfp4_grouped_amax(1, nv.NVFP4_IN_BF16, 4, 4, 1, 0, 1, None, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "num_groups" in nv.nvfp4_last_error()
    st = L.nvfp4_amax(1, nv.NVFP4_IN_BF16, 4, 4, None, None, None, None, None)
    assert st == nv.NVFP4_ERR_INVALID


def test_gemm_host_validation_without_gpu(lib_path):
    """nvfp4_gemm's argument checks and workspace size are host-only."""
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    # scales in the layout of their TMEM copies: 8 KB per 128 lines of A and 16 KB per
    # 256 lines of B, per K tile of 256 (3 and 2 tiles, 32 K tiles)
    assert nv.nvfp4_gemm_workspace_size(300, 500, 8192) == 3 * 32 * 8192 + 2 * 32 * 16384
    assert nv.nvfp4_gemm_workspace_size(0, 500, 8192) == 0
    ok = nv._COperand(256, 256, 256, nv.NVFP4_ROW_SCALED, 448.0)
    bad_bound = nv._COperand(256, 256, 256, nv.NVFP4_ROW_SCALED, 500.0)
    unaligned = nv._COperand(257, 256, 256, nv.NVFP4_PER_TENSOR, 256.0)
    R = ctypes.byref
    st = L.nvfp4_gemm(R(ok), R(bad_bound), 4, 4, 64, 256, nv.NVFP4_OUT_BF16, 256, 1 << 20, None)
    assert st == nv.NVFP4_ERR_INVALID and "bound" in nv.nvfp4_last_error()
    st = L.nvfp4_gemm(R(ok), R(ok), 4, 4, 48, 256, nv.NVFP4_OUT_BF16, 256, 1 << 20, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "multiple of 32" in nv.nvfp4_last_error()
    st = L.nvfp4_gemm(R(ok), R(unaligned), 4, 4, 64, 256, nv.NVFP4_OUT_FP32, 256, 1 << 20, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "aligned" in nv.nvfp4_last_error()
    st = L.nvfp4_gemm(R(ok), R(ok), 4, 4, 64, 256, nv.NVFP4_OUT_FP32, 256, 16, None)
    assert st == nv.NVFP4_ERR_INVALID and "workspace" in nv.nvfp4_last_error()
    st = L.nvfp4_gemm(R(ok), R(ok), 4, 4, 64, 256, 5, 256, 1 << 20, None)
    assert st == nv.NVFP4_ERR_INVALID and "out_dtype" in nv.nvfp4_last_error()
    st = L.nvfp4_gemm(None, R(ok), 4, 4, 64, 256, nv.NVFP4_OUT_FP32, 256, 1 << 20, None)
    assert st == nv.NVFP4_ERR_INVALID


def test_gemm_static_ws_rejects_oversize_without_gpu(lib_path):
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    ok = nv._COperand(256, 256, 256, nv.NVFP4_ROW_SCALED, 448.0)
    R = ctypes.byref
    assert nv.nvfp4_gemm_workspace_size(65536, 65536, 65536) > nv.NVFP4_GEMM_STATIC_WS_BYTES
    st = L.nvfp4_gemm_static_ws(R(ok), R(ok), 65536, 65536, 65536, 256, nv.NVFP4_OUT_BF16, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "static workspace" in nv.nvfp4_last_error()


def test_rht_host_validation_without_gpu(lib_path):
    """The transform's argument checks run before any CUDA call."""
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    R = ctypes.byref
    st = L.nvfp4_rht16(256, nv.NVFP4_IN_BF16, 24, 8, 0, 512, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "multiple of 16" in nv.nvfp4_last_error()
    st = L.nvfp4_rht16(256, nv.NVFP4_IN_BF16, 32, 8, 0x10000, 512, None)
    assert st == nv.NVFP4_ERR_INVALID and "sign_mask" in nv.nvfp4_last_error()
    st = L.nvfp4_rht16(256, 7, 32, 8, 0, 512, None)
    assert st == nv.NVFP4_ERR_INVALID and "dtype" in nv.nvfp4_last_error()
    st = L.nvfp4_rht16(256, nv.NVFP4_IN_BF16, 32, 8, 0, 256, None)
    assert st == nv.NVFP4_ERR_INVALID and "FP32" in nv.nvfp4_last_error()
    st = L.nvfp4_rht16(256, nv.NVFP4_IN_FP32, 32, 8, 0, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "y is NULL" in nv.nvfp4_last_error()
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
    col = nv._COut(1024, 2048, 4096, None)
    tiles = nv.Config(nv.NVFP4_PER_TENSOR, 448.0, 0, 1)  # 16x16 blocks need the workspace
    st = L.nvfp4_quantize_columnwise_rht(256, nv.NVFP4_IN_BF16, 32, 8, 0, R(tiles), R(col), 512,
                                         4 * 32 * 8 - 4, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "workspace" in nv.nvfp4_last_error()
    bad = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 1)
    st = L.nvfp4_quantize_columnwise_rht(256, nv.NVFP4_IN_BF16, 32, 8, 0, R(bad), R(col), 512,
                                         4 * 32 * 8, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "16x16" in nv.nvfp4_last_error()
    st = L.nvfp4_quantize_columnwise_rht(256, nv.NVFP4_IN_BF16, 40, 8, 0, R(cfg), R(col), 512,
                                         4 * 40 * 8, None, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED


def test_both_rht_host_validation_without_gpu(lib_path):
    """The two-direction transform quantize rejects what it does not cover before any
    CUDA call: 16x16 blocks, rows not a multiple of 16, x rows not 16-byte aligned, a
    missing direction."""
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    R = ctypes.byref
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
    row = nv._COut(1024, 2048, 4096, None)
    col = nv._COut(8192, 16384, 32768, None)
    st = L.nvfp4_quantize_both_rht(256, nv.NVFP4_IN_BF16, 40, 64, 0, R(cfg), R(row), R(col),
                                   None, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "multiple of 16" in nv.nvfp4_last_error()
    tiles = nv.Config(nv.NVFP4_PER_TENSOR, 448.0, 0, 1)
    st = L.nvfp4_quantize_both_rht(256, nv.NVFP4_IN_BF16, 32, 64, 0, R(tiles), R(row), R(col),
                                   None, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "1x16" in nv.nvfp4_last_error()
    st = L.nvfp4_quantize_both_rht(256, nv.NVFP4_IN_BF16, 32, 64, 0, R(cfg), None, R(col),
                                   None, None)
    assert st == nv.NVFP4_ERR_INVALID
    st = L.nvfp4_quantize_both_rht(256, nv.NVFP4_IN_BF16, 32, 36, 0, R(cfg), R(row), R(col),
                                   None, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "16-byte" in nv.nvfp4_last_error()
    st = L.nvfp4_quantize_both_rht(264, nv.NVFP4_IN_FP32, 32, 64, 0, R(cfg), R(row), R(col),
                                   None, None)
    assert st == nv.NVFP4_ERR_UNSUPPORTED and "16-byte" in nv.nvfp4_last_error()
    st = L.nvfp4_quantize_both_rht(256, nv.NVFP4_IN_BF16, 32, 64, 0x10000, R(cfg), R(row),
                                   R(col), None, None)
    assert st == nv.NVFP4_ERR_INVALID and "sign_mask" in nv.nvfp4_last_error()


def test_overlap_and_selftest_validation_without_gpu(lib_path):
    """Overlapping buffers of the transform and the self-test's limits are rejected on
    the host, before any CUDA call."""
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    R = ctypes.byref
    base = 1 << 20
    # FP32 x of 32 x 8 values is 1 KB: a y 4 bytes further overlaps it, y == x does not count
    st = L.nvfp4_rht16(base, nv.NVFP4_IN_FP32, 32, 8, 0, base + 4, None)
    assert st == nv.NVFP4_ERR_INVALID and "overlaps" in nv.nvfp4_last_error()
    # BF16 x is 512 bytes: y inside it, or ending inside it, is rejected
    st = L.nvfp4_rht16(base, nv.NVFP4_IN_BF16, 32, 8, 0, base + 256, None)
    assert st == nv.NVFP4_ERR_INVALID and "overlaps" in nv.nvfp4_last_error()
    st = L.nvfp4_rht16(base, nv.NVFP4_IN_BF16, 32, 8, 0, base - 1020, None)
    assert st == nv.NVFP4_ERR_INVALID and "overlaps" in nv.nvfp4_last_error()
    # adjacent buffers pass the checks (the call then needs a device)
    for y in (base + 512, base - 1024):
        st = L.nvfp4_rht16(base, nv.NVFP4_IN_BF16, 32, 8, 0, y, None)
        assert st != nv.NVFP4_ERR_INVALID, nv.nvfp4_last_error()
    st = L.nvfp4_rht16(base, nv.NVFP4_IN_FP32, 32, 8, 0, base, None)
    assert st != nv.NVFP4_ERR_INVALID, nv.nvfp4_last_error()
    # 16x16 transform workspace against x and each output
    tiles = nv.Config(nv.NVFP4_PER_TENSOR, 448.0, 0, 1)
    ws = 1 << 24
    need = 4 * 32 * 8
    for col in (nv._COut(ws + 8, 2 << 20, 3 << 20, None),       # codes inside the workspace
                nv._COut(2 << 20, ws + need - 1, 3 << 20, None),  # scales start on its last byte
                nv._COut(2 << 20, 3 << 20, ws, None)):           # amax at its start
        st = L.nvfp4_quantize_columnwise_rht(base, nv.NVFP4_IN_BF16, 32, 8, 0, R(tiles), R(col),
                                             ws, need, None, None)
        assert st == nv.NVFP4_ERR_INVALID and "overlaps" in nv.nvfp4_last_error()
    col = nv._COut(2 << 20, 3 << 20, 4 << 20, None)
    st = L.nvfp4_quantize_columnwise_rht(ws + 16, nv.NVFP4_IN_BF16, 32, 8, 0, R(tiles), R(col),
                                         ws, need, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "overlaps" in nv.nvfp4_last_error()
    # the bounded-wait self-test: limit within [0, 1 s], an output pointer
    st = L.nvfp4_selftest_wait_timeout(2_000_000_000, base, None)
    assert st == nv.NVFP4_ERR_INVALID and "limit_ns" in nv.nvfp4_last_error()
    st = L.nvfp4_selftest_wait_timeout(-1, base, None)
    assert st == nv.NVFP4_ERR_INVALID
    st = L.nvfp4_selftest_wait_timeout(1000, None, None)
    assert st == nv.NVFP4_ERR_INVALID and "out" in nv.nvfp4_last_error()


def test_scale_division_selftest_validation_without_gpu(lib_path):
    import nvfp4_precision_quantization_gb300 as nv
    L = nv.load_library()
    assert L.nvfp4_selftest_scale_division(1 << 20, -1, 1 << 21, None) == nv.NVFP4_ERR_INVALID
    assert L.nvfp4_selftest_scale_division(None, 4, 1 << 21, None) == nv.NVFP4_ERR_INVALID
    assert L.nvfp4_selftest_scale_division(1 << 20, 4, None, None) == nv.NVFP4_ERR_INVALID
    assert L.nvfp4_selftest_scale_division(None, 0, None, None) == nv.NVFP4_OK
