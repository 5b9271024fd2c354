"""NVFP4 quantize / dequantize on GB300 (sm_103a) -- Python binding of libnvfp4.

Thin ctypes layer over the C ABI declared in ``include/nvfp4.h``: the functions
keep the C names and only marshal arguments (torch tensors -> device pointers,
the current torch stream -> cudaStream_t).  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
importing a function without the compiled library raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
import os
import platform
from dataclasses import dataclass
from typing import Optional

import torch

__all__ = [
    "NVFP4_OK", "NVFP4_IN_BF16", "NVFP4_IN_FP32", "NVFP4_OUT_BF16", "NVFP4_OUT_FP32",
    "NVFP4_PER_TENSOR", "NVFP4_ROW_SCALED", "NVFP4_DEVICE_TIMEOUT", "NVFP4_DEVICE_BAD_GROUPS",
    "Config", "Out", "NVFP4Error", "load_library", "library_path",
    "nvfp4_amax", "nvfp4_quantize_rowwise", "nvfp4_quantize_columnwise", "nvfp4_quantize_both",
    "nvfp4_dequantize", "nvfp4_grouped_amax", "nvfp4_grouped_quantize_rowwise",
    "nvfp4_grouped_quantize_rowwise_padded", "nvfp4_grouped_quantize_columnwise",
    "nvfp4_last_error", "nvfp4_device_status", "nvfp4_selftest_convert",
    "nvfp4_selftest_wait_timeout", "nvfp4_selftest_scale_division",
    "nvfp4_gemm_workspace_size", "nvfp4_gemm", "nvfp4_gemm_static_ws", "Operand",
    "nvfp4_grouped_gemm_workspace_size", "nvfp4_grouped_gemm", "nvfp4_grouped_gemm_wgrad",
    "NVFP4_GEMM_STATIC_WS_BYTES", "alloc_out", "EXPORTED_SYMBOLS", "nvfp4_rht16",
    "nvfp4_quantize_columnwise_rht", "nvfp4_quantize_both_rht",
    "nvfp4_grouped_quantize_columnwise_rht",
]

NVFP4_OK = 0
NVFP4_ERR_INVALID = 1
NVFP4_ERR_UNSUPPORTED = 2
NVFP4_ERR_CUDA = 3
NVFP4_ERR_TIMEOUT = 4
NVFP4_IN_BF16 = 0
NVFP4_IN_FP32 = 1
NVFP4_OUT_BF16 = 0
NVFP4_OUT_FP32 = 1
NVFP4_PER_TENSOR = 0
NVFP4_ROW_SCALED = 1
NVFP4_DEVICE_TIMEOUT = 1
NVFP4_DEVICE_BAD_GROUPS = 2
NVFP4_GEMM_STATIC_WS_BYTES = 64 << 20

EXPORTED_SYMBOLS = (
    "nvfp4_amax", "nvfp4_quantize_rowwise", "nvfp4_quantize_columnwise", "nvfp4_quantize_both",
    "nvfp4_dequantize", "nvfp4_grouped_amax", "nvfp4_grouped_quantize_rowwise",
    "nvfp4_grouped_quantize_rowwise_padded", "nvfp4_grouped_quantize_columnwise",
    "nvfp4_last_error", "nvfp4_device_status", "nvfp4_selftest_convert",
    "nvfp4_selftest_wait_timeout", "nvfp4_selftest_scale_division",
    "nvfp4_gemm_workspace_size", "nvfp4_gemm", "nvfp4_gemm_static_ws",
    "nvfp4_grouped_gemm_workspace_size", "nvfp4_grouped_gemm", "nvfp4_grouped_gemm_wgrad",
    "nvfp4_rht16", "nvfp4_quantize_columnwise_rht", "nvfp4_quantize_both_rht",
    "nvfp4_grouped_quantize_columnwise_rht",
)

_HERE = os.path.dirname(os.path.abspath(__file__))


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"nvfp4 status {status}: {message}")
        self.status = status


class Config(C.Structure):
    """nvfp4_config: mode (PER_TENSOR / ROW_SCALED), bound (448 or 256),
    four_over_six (0/1), block_2d (0: 1x16, 1: 16x16)."""
    _fields_ = [("mode", C.c_int32), ("bound", C.c_float), ("four_over_six", C.c_int32),
                ("block_2d", C.c_int32)]


class _COut(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("amax", C.c_void_p),
                ("amax_in", C.c_void_p)]


@dataclass
class Out:
    """One output direction: codes [lines][ceil(n/2)] uint8, scales
    [lines][ceil(n/16)] uint8, amax [lines] or [1] float32, optional amax_in."""
    codes: torch.Tensor
    scales: torch.Tensor
    amax: torch.Tensor
    amax_in: Optional[torch.Tensor] = None

    def _c(self) -> _COut:
        return _COut(_ptr(self.codes), _ptr(self.scales), _ptr(self.amax), _ptr(self.amax_in))

    def as_operand(self, mode: int, bound: float) -> "Operand":
        return Operand(self.codes, self.scales, self.amax, mode, bound)


def library_path() -> str:
    return os.path.join(_HERE, f"libnvfp4_{platform.machine()}.so")


_lib = None


def load_library():
    """Load libnvfp4 (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libnvfp4 is not built ({path} missing); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = C.CDLL(path)
    vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
    sig = {
        "nvfp4_amax": [vp, i32, i64, i64, vp, vp, vp, vp, vp],
        "nvfp4_quantize_rowwise": [vp, i32, i64, i64, vp, vp, vp, vp],
        "nvfp4_quantize_columnwise": [vp, i32, i64, i64, vp, vp, vp, vp],
        "nvfp4_quantize_both": [vp, i32, i64, i64, vp, vp, vp, vp, vp],
        "nvfp4_dequantize": [vp, vp, vp, i32, i64, i64, f32, vp, i32, vp],
        "nvfp4_grouped_amax": [vp, i32, i64, i64, vp, i32, vp, vp, vp, vp],
        "nvfp4_grouped_quantize_rowwise": [vp, i32, i64, i64, vp, i32, vp, vp, vp, vp, vp],
        "nvfp4_grouped_quantize_rowwise_padded": [vp, i32, i64, i64, vp, vp, i32, i64, vp, vp,
                                                  vp, vp, vp],
        "nvfp4_grouped_quantize_columnwise": [vp, i32, i64, i64, vp, i32, vp, vp, vp, vp],
        "nvfp4_device_status": [C.POINTER(C.c_int32), i32],
        "nvfp4_selftest_convert": [vp, i64, vp, vp, vp],
        "nvfp4_selftest_wait_timeout": [i64, vp, vp],
        "nvfp4_selftest_scale_division": [vp, i64, vp, vp],
        "nvfp4_gemm_workspace_size": [i64, i64, i64, C.POINTER(C.c_uint64)],
        "nvfp4_gemm": [vp, vp, i64, i64, i64, vp, i32, vp, C.c_uint64, vp],
        "nvfp4_gemm_static_ws": [vp, vp, i64, i64, i64, vp, i32, vp],
        "nvfp4_grouped_gemm_workspace_size": [i64, i64, i64, i32, C.POINTER(C.c_uint64)],
        "nvfp4_grouped_gemm": [vp, vp, vp, i32, i64, i64, i64, vp, i32, vp, C.c_uint64, vp],
        "nvfp4_grouped_gemm_wgrad": [vp, vp, vp, i32, i64, i64, i64, vp, i32, vp, C.c_uint64,
                                     vp],
        "nvfp4_rht16": [vp, i32, i64, i64, C.c_uint32, vp, vp],
        "nvfp4_quantize_columnwise_rht": [vp, i32, i64, i64, C.c_uint32, vp, vp, vp, C.c_uint64,
                                          vp, vp],
        "nvfp4_quantize_both_rht": [vp, i32, i64, i64, C.c_uint32, vp, vp, vp, vp, vp],
        "nvfp4_grouped_quantize_columnwise_rht": [vp, i32, i64, i64, vp, i32, C.c_uint32, vp, vp,
                                                  vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_int
    L.nvfp4_last_error.argtypes = []
    L.nvfp4_last_error.restype = C.c_char_p
    _lib = L
    return L


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != NVFP4_OK:
        raise NVFP4Error(status, nvfp4_last_error())


def _in_dtype(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return NVFP4_IN_BF16
    if x.dtype == torch.float32:
        return NVFP4_IN_FP32
    raise TypeError(f"x must be bfloat16 or float32, got {x.dtype}")


def _matrix(x: torch.Tensor):
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    return x.shape[0], x.shape[1]


def nvfp4_last_error() -> str:
    return load_library().nvfp4_last_error().decode()


def nvfp4_amax(x: torch.Tensor, row_amax=None, col_amax=None, tensor_amax=None, noop=None,
               stream=None) -> None:
    rows, cols = _matrix(x)
    _check(load_library().nvfp4_amax(_ptr(x), _in_dtype(x), rows, cols, _ptr(row_amax),
                                     _ptr(col_amax), _ptr(tensor_amax), _ptr(noop),
                                     _stream(stream)))


def nvfp4_quantize_rowwise(x: torch.Tensor, cfg: Config, row: Out, noop=None, stream=None):
    rows, cols = _matrix(x)
    r = row._c()
    _check(load_library().nvfp4_quantize_rowwise(_ptr(x), _in_dtype(x), rows, cols,
                                                 C.byref(cfg), C.byref(r), _ptr(noop),
                                                 _stream(stream)))


def nvfp4_quantize_columnwise(x: torch.Tensor, cfg: Config, col: Out, noop=None, stream=None):
    rows, cols = _matrix(x)
    c = col._c()
    _check(load_library().nvfp4_quantize_columnwise(_ptr(x), _in_dtype(x), rows, cols,
                                                    C.byref(cfg), C.byref(c), _ptr(noop),
                                                    _stream(stream)))


def nvfp4_rht16(x: torch.Tensor, sign_mask: int, y: torch.Tensor, stream=None) -> None:
    """y (FP32, x's shape) = the random Hadamard transform of x along its rows, per
    column and per 16-row block, with the given 16-bit sign mask."""
    rows, cols = _matrix(x)
    if y.dtype != torch.float32 or tuple(y.shape) != (rows, cols) or not y.is_contiguous():
        raise ValueError("y must be a contiguous float32 tensor of x's shape")
    _check(load_library().nvfp4_rht16(_ptr(x), _in_dtype(x), rows, cols, sign_mask, _ptr(y),
                                      _stream(stream)))


def nvfp4_quantize_columnwise_rht(x: torch.Tensor, sign_mask: int, cfg: Config, col: Out,
                                  workspace: Optional[torch.Tensor] = None, noop=None,
                                  stream=None) -> None:
    """Columnwise quantization of the transformed x.  1x16 blocks: fused, no
    workspace.  16x16 blocks: workspace, a device buffer of at least 4 * rows * cols
    bytes, receives the transformed operand."""
    rows, cols = _matrix(x)
    c = col._c()
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().nvfp4_quantize_columnwise_rht(
        _ptr(x), _in_dtype(x), rows, cols, sign_mask, C.byref(cfg), C.byref(c), _ptr(workspace),
        nbytes, _ptr(noop), _stream(stream)))


def nvfp4_grouped_quantize_columnwise_rht(x: torch.Tensor, group_ends: torch.Tensor,
                                          sign_mask: int, cfg: Config, col: Out, noop=None,
                                          stream=None) -> None:
    """Grouped columnwise quantization of the transformed x (each group's amax)."""
    rows, cols = _matrix(x)
    c = col._c()
    _check(load_library().nvfp4_grouped_quantize_columnwise_rht(
        _ptr(x), _in_dtype(x), rows, cols, _ptr(group_ends), group_ends.numel(), sign_mask,
        C.byref(cfg), C.byref(c), _ptr(noop), _stream(stream)))


def nvfp4_quantize_both_rht(x: torch.Tensor, sign_mask: int, cfg: Config, row: Out, col: Out,
                            noop=None, stream=None) -> None:
    """Rowwise quantization of x and columnwise quantization of the transformed x in
    one encode pass (1x16 blocks)."""
    rows, cols = _matrix(x)
    r, c = row._c(), col._c()
    _check(load_library().nvfp4_quantize_both_rht(
        _ptr(x), _in_dtype(x), rows, cols, sign_mask, C.byref(cfg), C.byref(r), C.byref(c),
        _ptr(noop), _stream(stream)))


def nvfp4_quantize_both(x: torch.Tensor, cfg: Config, row: Out, col: Out, noop=None,
                        stream=None):
    rows, cols = _matrix(x)
    r, c = row._c(), col._c()
    _check(load_library().nvfp4_quantize_both(_ptr(x), _in_dtype(x), rows, cols, C.byref(cfg),
                                              C.byref(r), C.byref(c), _ptr(noop),
                                              _stream(stream)))


def nvfp4_dequantize(codes, scales, amax, mode: int, rows: int, cols: int, bound: float,
                     out: torch.Tensor, stream=None) -> None:
    if out.dtype == torch.bfloat16:
        od = NVFP4_OUT_BF16
    elif out.dtype == torch.float32:
        od = NVFP4_OUT_FP32
    else:
        raise TypeError("out must be bfloat16 or float32")
    _check(load_library().nvfp4_dequantize(_ptr(codes), _ptr(scales), _ptr(amax), mode, rows,
                                           cols, bound, _ptr(out), od, _stream(stream)))


def nvfp4_grouped_amax(x: torch.Tensor, group_ends: torch.Tensor, group_amax: torch.Tensor,
                       row_amax_expanded=None, noop=None, stream=None) -> None:
    rows, cols = _matrix(x)
    _check(load_library().nvfp4_grouped_amax(_ptr(x), _in_dtype(x), rows, cols,
                                             _ptr(group_ends), int(group_ends.numel()),
                                             _ptr(group_amax), _ptr(row_amax_expanded),
                                             _ptr(noop), _stream(stream)))


def nvfp4_grouped_quantize_rowwise(x: torch.Tensor, group_ends: torch.Tensor, cfg: Config,
                                   row: Out, group_amax=None, noop=None, stream=None) -> None:
    rows, cols = _matrix(x)
    r = row._c()
    _check(load_library().nvfp4_grouped_quantize_rowwise(
        _ptr(x), _in_dtype(x), rows, cols, _ptr(group_ends), int(group_ends.numel()),
        C.byref(cfg), C.byref(r), _ptr(group_amax), _ptr(noop), _stream(stream)))


def nvfp4_grouped_quantize_rowwise_padded(x: torch.Tensor, ragged_ends: torch.Tensor,
                                          padded_ends: torch.Tensor, padded_rows: int,
                                          cfg: Config, row: Out, group_amax: torch.Tensor,
                                          noop=None, stream=None) -> None:
    tokens, cols = _matrix(x)
    r = row._c()
    _check(load_library().nvfp4_grouped_quantize_rowwise_padded(
        _ptr(x), _in_dtype(x), tokens, cols, _ptr(ragged_ends), _ptr(padded_ends),
        int(ragged_ends.numel()), int(padded_rows), C.byref(cfg), C.byref(r), _ptr(group_amax),
        _ptr(noop), _stream(stream)))


def nvfp4_grouped_quantize_columnwise(x: torch.Tensor, group_ends: torch.Tensor, cfg: Config,
                                      col: Out, noop=None, stream=None) -> None:
    rows, cols = _matrix(x)
    c = col._c()
    _check(load_library().nvfp4_grouped_quantize_columnwise(
        _ptr(x), _in_dtype(x), rows, cols, _ptr(group_ends), int(group_ends.numel()),
        C.byref(cfg), C.byref(c), _ptr(noop), _stream(stream)))


def nvfp4_device_status(reset: bool = False, raise_on_timeout: bool = False) -> int:
    """The device status word's NVFP4_DEVICE_* bits.  The C call returns
    NVFP4_ERR_TIMEOUT when the timeout bit is set; that raises here only with
    raise_on_timeout, else the bits are returned as for any other state."""
    v = C.c_int32(0)
    rc = load_library().nvfp4_device_status(C.byref(v), int(reset))
    if rc != NVFP4_ERR_TIMEOUT or raise_on_timeout:
        _check(rc)
    return v.value


def nvfp4_selftest_scale_division(S: torch.Tensor, e_out: torch.Tensor, stream=None) -> None:
    """e_out[i, s8] = the encode kernels' fl(S[i] / decode(s8)) for s8 = 0 .. 126."""
    if S.dtype != torch.float32 or not S.is_contiguous():
        raise TypeError("S must be contiguous float32")
    if e_out.dtype != torch.float32 or e_out.numel() != S.numel() * 127:
        raise TypeError("e_out must be float32 with S.numel() * 127 elements")
    _check(load_library().nvfp4_selftest_scale_division(_ptr(S), S.numel(), _ptr(e_out),
                                                        _stream(stream)))


def nvfp4_selftest_wait_timeout(limit_ns: int, out: torch.Tensor, stream=None) -> None:
    """Run the bounded-wait self-test: a wait that nothing completes, given up after
    limit_ns nanoseconds (out: one device uint32, left untouched when it gives up)."""
    if out.dtype not in (torch.int32, torch.uint32) or out.numel() < 1:
        raise TypeError("out must hold at least one 32-bit integer")
    _check(load_library().nvfp4_selftest_wait_timeout(int(limit_ns), _ptr(out), _stream(stream)))


def nvfp4_selftest_convert(x: torch.Tensor, e2m1_out=None, e4m3_out=None, stream=None) -> None:
    if x.dtype != torch.float32 or not x.is_contiguous():
        raise TypeError("x must be contiguous float32")
    _check(load_library().nvfp4_selftest_convert(_ptr(x), x.numel(), _ptr(e2m1_out),
                                                 _ptr(e4m3_out), _stream(stream)))


class _COperand(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("amax", C.c_void_p),
                ("mode", C.c_int32), ("bound", C.c_float)]


@dataclass
class Operand:
    """One nvfp4_gemm operand (nvfp4_operand): K-major codes [lines][k/2], scales
    [lines][k/16], amax [lines] (ROW_SCALED) or [1] (PER_TENSOR), the bound it was
    quantized with.  Out.as_operand() builds one from a quantize output."""
    codes: torch.Tensor
    scales: torch.Tensor
    amax: torch.Tensor
    mode: int
    bound: float

    def _c(self) -> _COperand:
        return _COperand(_ptr(self.codes), _ptr(self.scales), _ptr(self.amax), self.mode,
                         self.bound)


def nvfp4_gemm_workspace_size(m: int, n: int, k: int) -> int:
    v = C.c_uint64(0)
    _check(load_library().nvfp4_gemm_workspace_size(m, n, k, C.byref(v)))
    return v.value


def nvfp4_gemm(a: Operand, b: Operand, d: torch.Tensor, workspace: Optional[torch.Tensor] = None,
               stream=None) -> None:
    """d [m][n] (bfloat16 or float32) = dequant(a) x dequant(b)^T on the tensor cores.
    workspace: uint8 device tensor of nvfp4_gemm_workspace_size(m, n, k) bytes (allocated
    here with torch if not given)."""
    if d.dim() != 2 or not d.is_contiguous():
        raise ValueError("d must be a contiguous 2-D tensor")
    if d.dtype == torch.bfloat16:
        od = NVFP4_OUT_BF16
    elif d.dtype == torch.float32:
        od = NVFP4_OUT_FP32
    else:
        raise TypeError("d must be bfloat16 or float32")
    m, n = d.shape
    k = a.codes.shape[1] * 2
    if a.codes.shape[0] != m or b.codes.shape[0] != n or b.codes.shape[1] * 2 != k:
        raise ValueError("operand shapes do not match d")
    need = nvfp4_gemm_workspace_size(m, n, k)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d.device)
    ca, cb = a._c(), b._c()
    _check(load_library().nvfp4_gemm(C.byref(ca), C.byref(cb), m, n, k, _ptr(d), od,
                                      _ptr(workspace), workspace.numel(), _stream(stream)))


def nvfp4_grouped_gemm_workspace_size(rows: int, n: int, k: int, num_groups: int) -> int:
    v = C.c_uint64(0)
    _check(load_library().nvfp4_grouped_gemm_workspace_size(rows, n, k, num_groups, C.byref(v)))
    return v.value


def nvfp4_grouped_gemm(a: Operand, b: Operand, group_ends: torch.Tensor, d: torch.Tensor,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """d [rows][n] = per group g: dequant(a rows of g) x dequant(b rows [g*n, (g+1)*n))^T.
    group_ends: device int64 [groups]; b.codes has groups * n rows."""
    if d.dim() != 2 or not d.is_contiguous():
        raise ValueError("d must be a contiguous 2-D tensor")
    if d.dtype == torch.bfloat16:
        od = NVFP4_OUT_BF16
    elif d.dtype == torch.float32:
        od = NVFP4_OUT_FP32
    else:
        raise TypeError("d must be bfloat16 or float32")
    rows, n = d.shape
    groups = int(group_ends.numel())
    k = a.codes.shape[1] * 2
    if a.codes.shape[0] != rows or b.codes.shape[0] != groups * n or b.codes.shape[1] * 2 != k:
        raise ValueError("operand shapes do not match d and the group count")
    need = nvfp4_grouped_gemm_workspace_size(rows, n, k, groups)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d.device)
    ca, cb = a._c(), b._c()
    _check(load_library().nvfp4_grouped_gemm(C.byref(ca), C.byref(cb), _ptr(group_ends), groups,
                                              rows, n, k, _ptr(d), od, _ptr(workspace),
                                              workspace.numel(), _stream(stream)))


def nvfp4_grouped_gemm_wgrad(a: Operand, b: Operand, group_ends: torch.Tensor, d: torch.Tensor,
                             workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """d [groups][m][n]: per group g, dequant(a) x dequant(b)^T over g's token range of K.
    a [m][tokens/2], b [n][tokens/2] (columnwise outputs); group_ends device int64."""
    if d.dim() != 3 or not d.is_contiguous():
        raise ValueError("d must be a contiguous 3-D tensor [groups][m][n]")
    if d.dtype == torch.bfloat16:
        od = NVFP4_OUT_BF16
    elif d.dtype == torch.float32:
        od = NVFP4_OUT_FP32
    else:
        raise TypeError("d must be bfloat16 or float32")
    groups, m, n = d.shape
    tokens = a.codes.shape[1] * 2
    if (groups != group_ends.numel() or a.codes.shape[0] != m or b.codes.shape[0] != n
            or b.codes.shape[1] * 2 != tokens):
        raise ValueError("operand shapes do not match d and the group count")
    need = nvfp4_gemm_workspace_size(m, n, tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=d.device)
    ca, cb = a._c(), b._c()
    _check(load_library().nvfp4_grouped_gemm_wgrad(C.byref(ca), C.byref(cb), _ptr(group_ends),
                                                    groups, m, n, tokens, _ptr(d), od,
                                                    _ptr(workspace), workspace.numel(),
                                                    _stream(stream)))


def nvfp4_gemm_static_ws(a: Operand, b: Operand, d: torch.Tensor, stream=None) -> None:
    """nvfp4_gemm with the library's static device workspace (no workspace argument)."""
    if d.dim() != 2 or not d.is_contiguous():
        raise ValueError("d must be a contiguous 2-D tensor")
    if d.dtype == torch.bfloat16:
        od = NVFP4_OUT_BF16
    elif d.dtype == torch.float32:
        od = NVFP4_OUT_FP32
    else:
        raise TypeError("d must be bfloat16 or float32")
    m, n = d.shape
    k = a.codes.shape[1] * 2
    if a.codes.shape[0] != m or b.codes.shape[0] != n or b.codes.shape[1] * 2 != k:
        raise ValueError("operand shapes do not match d")
    ca, cb = a._c(), b._c()
    _check(load_library().nvfp4_gemm_static_ws(C.byref(ca), C.byref(cb), m, n, k, _ptr(d), od,
                                                _stream(stream)))


def alloc_out(lines: int, n: int, amax_len: int, device="cuda", fill=None) -> Out:
    """Allocate one output direction with torch (codes, scales, amax)."""
    codes = torch.empty(lines, (n + 1) // 2, dtype=torch.uint8, device=device)
    scales = torch.empty(lines, (n + 15) // 16, dtype=torch.uint8, device=device)
    amax = torch.empty(amax_len, dtype=torch.float32, device=device)
    if fill is not None:
        codes.fill_(fill)
        scales.fill_(fill)
    return Out(codes, scales, amax)
