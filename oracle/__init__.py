"""CPU oracle for NVFP4 quantize / dequantize -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it and never falls back to it.

This module marshals numpy arrays into the plain C oracle in
``nvfp4_oracle.c``; every step of the method lives there, one FP32 operation
at a time.  BF16 arrays are passed around as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

PER_TENSOR = 0
ROW_SCALED = 1


def lib():
    global _lib
    if _lib is None:
        # NVFP4_ORACLE_LIBRARY lets the mutation tests load a deliberately broken copy
        path = os.environ.get("NVFP4_ORACLE_LIBRARY") or _build.build()
        L = C.CDLL(path)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
        vp = C.c_void_p
        i64 = C.c_int64
        L.oracle_bf16_to_f32.restype = C.c_float
        L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
        L.oracle_f32_to_bf16.restype = C.c_uint16
        L.oracle_f32_to_bf16.argtypes = [C.c_float]
        L.oracle_e2m1_decode.restype = C.c_float
        L.oracle_e2m1_decode.argtypes = [C.c_uint8]
        L.oracle_e2m1_encode.restype = C.c_uint8
        L.oracle_e2m1_encode.argtypes = [C.c_float]
        L.oracle_e4m3_decode.restype = C.c_float
        L.oracle_e4m3_decode.argtypes = [C.c_uint8]
        L.oracle_e4m3_encode.restype = C.c_uint8
        L.oracle_e4m3_encode.argtypes = [C.c_float]
        L.oracle_e2m1_encode_array.restype = None
        L.oracle_e2m1_encode_array.argtypes = [f32p, i64, u8p]
        L.oracle_e4m3_encode_array.restype = None
        L.oracle_e4m3_encode_array.argtypes = [f32p, i64, u8p]
        L.oracle_bf16_to_f32_array.restype = None
        L.oracle_bf16_to_f32_array.argtypes = [u16p, i64, f32p]
        L.oracle_fp_contract_probe.restype = C.c_float
        L.oracle_fp_contract_probe.argtypes = [C.c_float] * 3
        L.oracle_global_scale.restype = C.c_float
        L.oracle_global_scale.argtypes = [C.c_float, C.c_float]
        L.oracle_quantize_line.restype = None
        L.oracle_quantize_line.argtypes = [f32p, i64, i64, C.c_float, C.c_float, C.c_int, u8p, u8p]
        L.oracle_amax.restype = None
        L.oracle_amax.argtypes = [f32p, i64, i64, vp, vp, vp]
        L.oracle_quantize.restype = C.c_int
        L.oracle_quantize.argtypes = [f32p, i64, i64, C.c_int, C.c_float, C.c_int, C.c_int,
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_dequantize.restype = None
        L.oracle_dequantize.argtypes = [u8p, u8p, f32p, C.c_int, i64, i64, C.c_float, vp, C.c_int]
        L.oracle_grouped_amax.restype = C.c_int
        L.oracle_grouped_amax.argtypes = [f32p, i64, i64, i64p, C.c_int, vp, vp, vp]
        L.oracle_grouped_quantize_rowwise.restype = C.c_int
        L.oracle_grouped_quantize_rowwise.argtypes = [f32p, i64, i64, i64p, C.c_int, C.c_int,
                                                      C.c_float, C.c_int, vp, vp, vp, vp, vp]
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        L.oracle_gemm.restype = None
        L.oracle_gemm.argtypes = [u8p, u8p, f32p, C.c_int, C.c_float, u8p, u8p, f32p, C.c_int,
                                  C.c_float, i64, i64, i64, f64p, vp]
        L.oracle_rht16.restype = C.c_int
        L.oracle_rht16.argtypes = [f32p, i64, i64, C.c_uint32, f32p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------
# Formats
# --------------------------------------------------------------------------

def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().oracle_bf16_to_f32_array(h.reshape(-1), h.size, out.reshape(-1))
    return out


def as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Step 1 of the recipe: read the input as FP32 (BF16 widening is exact)."""
    if dtype == "bf16":
        return bf16_to_f32(x)
    if dtype == "fp32":
        return _f32(x)
    raise ValueError(dtype)


def e2m1_encode(y) -> np.ndarray:
    y = _f32(y)
    out = np.empty(y.shape, np.uint8)
    lib().oracle_e2m1_encode_array(y.reshape(-1), y.size, out.reshape(-1))
    return out


def e2m1_decode(c) -> np.ndarray:
    L = lib()
    c = np.asarray(c, dtype=np.uint8)
    return np.array([L.oracle_e2m1_decode(int(v)) for v in c.reshape(-1)],
                    np.float32).reshape(c.shape)


def e4m3_encode(s) -> np.ndarray:
    s = _f32(s)
    out = np.empty(s.shape, np.uint8)
    lib().oracle_e4m3_encode_array(s.reshape(-1), s.size, out.reshape(-1))
    return out


def e4m3_decode(s) -> np.ndarray:
    L = lib()
    s = np.asarray(s, dtype=np.uint8)
    return np.array([L.oracle_e4m3_decode(int(v)) for v in s.reshape(-1)],
                    np.float32).reshape(s.shape)


def f32_to_bf16(f) -> np.ndarray:
    L = lib()
    f = _f32(f)
    return np.array([L.oracle_f32_to_bf16(float(v)) for v in f.reshape(-1)],
                    np.uint16).reshape(f.shape)


def global_scale(amax: float, bound: float) -> float:
    return lib().oracle_global_scale(amax, bound)


# --------------------------------------------------------------------------
# amax / quantize / dequantize / grouped
# --------------------------------------------------------------------------

def amax(x: np.ndarray, dtype: str = "fp32"):
    """Return (row_amax [rows], col_amax [cols], tensor_amax float)."""
    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    ra = np.empty(rows, np.float32)
    ca = np.empty(cols, np.float32)
    t = np.empty(1, np.float32)
    lib().oracle_amax(xf, rows, cols, _ptr(ra), _ptr(ca), _ptr(t))
    return ra, ca, float(t[0])


def quantize_line(values, amax_value: float, bound: float = 448.0, four_over_six: bool = False):
    """Quantize one line (a row, or a column read as a vector) with 1x16 blocks."""
    v = _f32(values).reshape(-1)
    n = v.size
    codes = np.zeros((n + 1) // 2, np.uint8)
    scales = np.zeros((n + 15) // 16, np.uint8)
    lib().oracle_quantize_line(v, n, 1, amax_value, bound, int(four_over_six), codes, scales)
    return codes, scales


def quantize(x: np.ndarray, dtype: str = "fp32", *, mode: int = ROW_SCALED, bound: float = 448.0,
             four_over_six: bool = False, block_2d: bool = False, rowwise: bool = True,
             columnwise: bool = True, row_amax_in=None, col_amax_in=None, noop=None, out=None):
    """Dense quantize.  Returns {"row": (codes, scales, amax), "col": (...)} for the
    requested directions.  ``out`` may supply pre-filled output arrays (the noop
    tests use sentinel-filled buffers)."""
    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    na_r = rows if mode == ROW_SCALED else 1
    na_c = cols if mode == ROW_SCALED else 1
    if out is None:
        out = {}
        if rowwise:
            out["row"] = (np.zeros((rows, (cols + 1) // 2), np.uint8),
                          np.zeros((rows, (cols + 15) // 16), np.uint8),
                          np.zeros(na_r, np.float32))
        if columnwise:
            out["col"] = (np.zeros((cols, (rows + 1) // 2), np.uint8),
                          np.zeros((cols, (rows + 15) // 16), np.uint8),
                          np.zeros(na_c, np.float32))
    r = out.get("row", (None, None, None))
    c = out.get("col", (None, None, None))
    rin = None if row_amax_in is None else _f32(row_amax_in)
    cin = None if col_amax_in is None else _f32(col_amax_in)
    nz = None if noop is None else np.array([noop], np.float32)
    rc = lib().oracle_quantize(xf, rows, cols, mode, bound, int(four_over_six), int(block_2d),
                               _ptr(rin), _ptr(cin), _ptr(r[0]), _ptr(r[1]), _ptr(r[2]),
                               _ptr(c[0]), _ptr(c[1]), _ptr(c[2]), _ptr(nz))
    if rc != 0:
        raise ValueError("oracle_quantize rejected the arguments")
    return out


def quantize_parallel(x: np.ndarray, dtype: str = "fp32", *, mode: int = ROW_SCALED,
                      bound: float = 448.0, four_over_six: bool = False, block_2d: bool = False,
                      rowwise: bool = True, columnwise: bool = True, threads: int | None = None,
                      strip: int = 64):
    """quantize() spread over host threads: the same C routine applied to strips of
    rows (rowwise output) and strips of columns (columnwise output), each strip given
    the amax the whole tensor has for its lines.

    No arithmetic is added.  Once every line's amax is known, each line (each 16x16
    tile with block_2d) is quantized on its own.  So a strip quantized with its
    lines' amax gives exactly the bytes that the whole-tensor call gives for those
    lines.  tests/test_oracle_parallel.py checks this equality.  The
    C calls release the GIL (ctypes), so the strips run on as many cores as there
    are threads.  Returns what quantize() returns."""
    import concurrent.futures as cf

    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    threads = threads or os.cpu_count() or 1
    strip = max(16, (strip // 16) * 16)  # whole 16-line blocks (16x16 tiles)
    ra, ca, t = amax(xf, "fp32")
    rs = mode == ROW_SCALED
    out = {}
    jobs = []
    if rowwise:
        out["row"] = (np.zeros((rows, (cols + 1) // 2), np.uint8),
                      np.zeros((rows, (cols + 15) // 16), np.uint8),
                      ra.copy() if rs else np.array([t], np.float32))
        rc, rsc, _ = out["row"]
        for r0 in range(0, rows, strip):
            r1 = min(rows, r0 + strip)
            jobs.append(("row", r0, r1, rc[r0:r1], rsc[r0:r1],
                         ra[r0:r1] if rs else np.array([t], np.float32)))
    if columnwise:
        out["col"] = (np.zeros((cols, (rows + 1) // 2), np.uint8),
                      np.zeros((cols, (rows + 15) // 16), np.uint8),
                      ca.copy() if rs else np.array([t], np.float32))
        cc, csc, _ = out["col"]
        for c0 in range(0, cols, strip):
            c1 = min(cols, c0 + strip)
            jobs.append(("col", c0, c1, cc[c0:c1], csc[c0:c1],
                         ca[c0:c1] if rs else np.array([t], np.float32)))

    def run(job):
        d, lo, hi, codes, scales, a = job
        L = lib()
        if d == "row":
            part = np.ascontiguousarray(xf[lo:hi])
            rc_ = L.oracle_quantize(part, hi - lo, cols, mode, bound, int(four_over_six),
                                    int(block_2d), _ptr(_f32(a)), None, _ptr(codes),
                                    _ptr(scales), None, None, None, None, None)
        else:
            part = np.ascontiguousarray(xf[:, lo:hi])
            rc_ = L.oracle_quantize(part, rows, hi - lo, mode, bound, int(four_over_six),
                                    int(block_2d), None, _ptr(_f32(a)), None, None, None,
                                    _ptr(codes), _ptr(scales), None, None)
        if rc_ != 0:
            raise ValueError("oracle_quantize rejected the arguments")

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, jobs))
    return out


def dequantize(codes, scales, amax_vec, *, row_scaled: bool, rows: int, cols: int,
               bound: float = 448.0, out_dtype: str = "fp32") -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8).reshape(-1)
    scales = np.ascontiguousarray(scales, np.uint8).reshape(-1)
    a = _f32(amax_vec).reshape(-1)
    if out_dtype == "bf16":
        out = np.empty((rows, cols), np.uint16)
    else:
        out = np.empty((rows, cols), np.float32)
    lib().oracle_dequantize(codes, scales, a, int(row_scaled), rows, cols, bound, _ptr(out),
                            int(out_dtype == "bf16"))
    return out


def grouped_amax(x: np.ndarray, dtype: str, group_ends, noop=None):
    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    ends = np.ascontiguousarray(group_ends, np.int64)
    g = np.zeros(max(len(ends), 1), np.float32)
    e = np.zeros(max(rows, 1), np.float32)
    nz = None if noop is None else np.array([noop], np.float32)
    rc = lib().oracle_grouped_amax(xf, rows, cols, ends, len(ends), _ptr(g), _ptr(e), _ptr(nz))
    if rc != 0:
        raise ValueError("invalid group ends")
    return g[:len(ends)], e[:rows]


def grouped_quantize_rowwise(x: np.ndarray, dtype: str, group_ends, *, mode: int = PER_TENSOR,
                             bound: float = 256.0, four_over_six: bool = True):
    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    ends = np.ascontiguousarray(group_ends, np.int64)
    codes = np.zeros((rows, (cols + 1) // 2), np.uint8)
    scales = np.zeros((rows, (cols + 15) // 16), np.uint8)
    ra = np.zeros(max(rows, 1), np.float32)
    ga = np.zeros(max(len(ends), 1), np.float32)
    rc = lib().oracle_grouped_quantize_rowwise(xf, rows, cols, ends, len(ends), mode, bound,
                                               int(four_over_six), _ptr(codes), _ptr(scales),
                                               _ptr(ra), _ptr(ga), None)
    if rc != 0:
        raise ValueError("invalid grouped arguments")
    return codes, scales, ra[:rows], ga[:len(ends)]


def gemm(a, b, *, with_abs: bool = False):
    """D = dequant(A) x dequant(B)^T in FP64 (the GEMM that consumes NVFP4 operands).

    a, b: dicts with "codes" [lines][k/2], "scales" [lines][k/16], "amax" ([lines] or
    [1]), "row_scaled" (bool) and "bound".  Returns D [m][n] (and, with with_abs, the
    per-element sum of |terms| that rounding bounds scale with)."""
    ac = np.ascontiguousarray(a["codes"], np.uint8)
    bc = np.ascontiguousarray(b["codes"], np.uint8)
    m, n, k = ac.shape[0], bc.shape[0], ac.shape[1] * 2
    assert bc.shape[1] * 2 == k and k % 16 == 0
    d = np.zeros((m, n), np.float64)
    da = np.zeros((m, n), np.float64) if with_abs else None
    lib().oracle_gemm(ac.reshape(-1), np.ascontiguousarray(a["scales"], np.uint8).reshape(-1),
                      _f32(a["amax"]).reshape(-1), int(a["row_scaled"]), float(a["bound"]),
                      bc.reshape(-1), np.ascontiguousarray(b["scales"], np.uint8).reshape(-1),
                      _f32(b["amax"]).reshape(-1), int(b["row_scaled"]), float(b["bound"]),
                      m, n, k, d, _ptr(da))
    return (d, da) if with_abs else d


def grouped_gemm(a, b, group_ends, n: int, *, with_abs: bool = False):
    """The per-expert GEMM of grouped tokens ("Add NVFP4 four-over-six grouped GEMM for
    MoE training", torchao PR #9, description): group g's rows of a, [e_{g-1}, e_g),
    times b's rows [g*n, (g+1)*n)^T, each block computed by gemm() above (no new
    arithmetic: only the slicing of the operands and of their amax).  b["amax"] holds
    [groups*n] per-line values (row_scaled) or [groups] per-expert values."""
    ends = np.asarray(group_ends, np.int64)
    rows = a["codes"].shape[0]
    d = np.zeros((rows, n), np.float64)
    da = np.zeros((rows, n), np.float64) if with_abs else None
    start = 0
    for g, e in enumerate(ends.tolist()):
        if e > start:
            ag = dict(a, codes=a["codes"][start:e], scales=a["scales"][start:e],
                      amax=a["amax"][start:e] if a["row_scaled"] else a["amax"])
            bam = b["amax"][g * n:(g + 1) * n] if b["row_scaled"] else b["amax"][g:g + 1]
            bg = dict(b, codes=b["codes"][g * n:(g + 1) * n], scales=b["scales"][g * n:(g + 1) * n],
                      amax=bam)
            r = gemm(ag, bg, with_abs=with_abs)
            if with_abs:
                d[start:e], da[start:e] = r
            else:
                d[start:e] = r
        start = e
    return (d, da) if with_abs else d


def grouped_gemm_wgrad(a, b, group_ends, *, with_abs: bool = False):
    """The per-expert weight-gradient GEMM: for group g, the token range [e_{g-1}, e_g)
    of K, d[g] = gemm() of a's and b's columns in that range (their codes, scales and
    group g's amax: [groups*lines] per line or [groups] per group).  Composition of the
    pinned gemm() above; no new arithmetic."""
    ends = np.asarray(group_ends, np.int64)
    m, n = a["codes"].shape[0], b["codes"].shape[0]
    G = len(ends)
    d = np.zeros((G, m, n), np.float64)
    da = np.zeros((G, m, n), np.float64) if with_abs else None

    def part(op, lines, g, s, e):
        am = op["amax"][g * lines:(g + 1) * lines] if op["row_scaled"] else op["amax"][g:g + 1]
        return dict(op, codes=op["codes"][:, s // 2:e // 2], scales=op["scales"][:, s // 16:e // 16],
                    amax=am)

    start = 0
    for g, e in enumerate(ends.tolist()):
        if e > start:
            r = gemm(part(a, m, g, start, e), part(b, n, g, start, e), with_abs=with_abs)
            if with_abs:
                d[g], da[g] = r
            else:
                d[g] = r
        start = e
    return (d, da) if with_abs else d


# --------------------------------------------------------------------------
# Random Hadamard transform of the columnwise operand (reading R14)
# --------------------------------------------------------------------------

def rht16(x: np.ndarray, dtype: str = "fp32", sign_mask: int = 0) -> np.ndarray:
    """y = (1/4) H16 diag(s) x along each column, per block of 16 rows, in FP32 (the
    oracle's reading R14; TE-3206's description names the transform, without a
    definition).  rows must be a multiple of 16."""
    xf = as_f32(x, dtype)
    rows, cols = xf.shape
    y = np.empty((rows, cols), np.float32)
    if lib().oracle_rht16(xf, rows, cols, sign_mask & 0xFFFF, y) != 0:
        raise ValueError("oracle_rht16: rows must be a multiple of 16")
    return y


def quantize_columnwise_rht(x: np.ndarray, dtype: str = "fp32", sign_mask: int = 0, *,
                            mode: int = ROW_SCALED, bound: float = 448.0,
                            four_over_six: bool = False, block_2d: bool = False):
    """The columnwise quantization of rht16(x): (codes, scales, amax)."""
    return quantize(rht16(x, dtype, sign_mask), "fp32", mode=mode, bound=bound,
                    four_over_six=four_over_six, block_2d=block_2d, rowwise=False)["col"]
