"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
(via the binding) and the oracle on the very same input bytes."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_precision_quantization_gb300 as nv
import oracle


def host_bits(x: torch.Tensor):
    """(numpy array, dtype tag) of a tensor's exact bytes for the oracle."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16), "bf16"
    return x.numpy().astype(np.float32, copy=False), "fp32"


def cfg(mode=nv.NVFP4_ROW_SCALED, bound=448.0, fos=False, b2d=False) -> nv.Config:
    return nv.Config(mode, bound, int(fos), int(b2d))


def gpu_quantize(x: torch.Tensor, c: nv.Config, rowwise=True, columnwise=True, noop=None,
                 row_amax_in=None, col_amax_in=None, fill=None, outs=None):
    rows, cols = x.shape
    rs = c.mode == nv.NVFP4_ROW_SCALED
    dev = x.device
    if outs is None:
        outs = {}
        if rowwise:
            outs["row"] = nv.alloc_out(rows, cols, rows if rs else 1, dev, fill)
        if columnwise:
            outs["col"] = nv.alloc_out(cols, rows, cols if rs else 1, dev, fill)
    if "row" in outs:
        outs["row"].amax_in = row_amax_in
    if "col" in outs:
        outs["col"].amax_in = col_amax_in
    if rowwise and columnwise:
        nv.nvfp4_quantize_both(x, c, outs["row"], outs["col"], noop=noop)
    elif rowwise:
        nv.nvfp4_quantize_rowwise(x, c, outs["row"], noop=noop)
    else:
        nv.nvfp4_quantize_columnwise(x, c, outs["col"], noop=noop)
    torch.cuda.synchronize()
    return outs


def to_np(o: nv.Out):
    return (o.codes.cpu().numpy(), o.scales.cpu().numpy(), o.amax.cpu().numpy())


def oracle_quantize(x: torch.Tensor, c: nv.Config, rowwise=True, columnwise=True,
                    row_amax_in=None, col_amax_in=None):
    xb, tag = host_bits(x)
    return oracle.quantize(xb, tag, mode=c.mode, bound=c.bound, four_over_six=bool(c.four_over_six),
                           block_2d=bool(c.block_2d), rowwise=rowwise, columnwise=columnwise,
                           row_amax_in=row_amax_in, col_amax_in=col_amax_in)


def assert_same(gpu: nv.Out, ref, what=""):
    g = to_np(gpu)
    for name, a, b in zip(("codes", "scales", "amax"), g, ref):
        a = np.asarray(a).reshape(np.asarray(b).shape)
        if name == "amax":
            eq = np.array_equal(a.view(np.uint32), np.asarray(b, np.float32).view(np.uint32))
        else:
            eq = np.array_equal(a, b)
        if not eq:
            bad = np.argwhere(a != b)
            raise AssertionError(f"{what} {name} differ at {len(bad)} places, first {bad[:5].tolist()}"
                                 f" gpu={a[tuple(bad[0])] if len(bad) else None}"
                                 f" oracle={b[tuple(bad[0])] if len(bad) else None}")
