"""The oracle's strip-parallel driver gives exactly the whole-tensor oracle's bytes.

quantize_parallel() only cuts the tensor into strips of lines and hands each strip
its lines' amax; these tests hold it to quantize() on shapes with ragged strips,
both modes, four-over-six, 16x16 tiles and FP32 input, so that the GPU tests and the
CPU baseline can use it in place of the single-threaded call.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _same(a, b):
    for d in a:
        for u, v in zip(a[d], b[d]):
            assert np.array_equal(np.asarray(u), np.asarray(v)), d


@pytest.mark.parametrize("shape", [(97, 200), (256, 130), (33, 17)])
@pytest.mark.parametrize("mode", [oracle.ROW_SCALED, oracle.PER_TENSOR])
@pytest.mark.parametrize("fos,bound", [(False, 448.0), (True, 256.0), (True, 448.0)])
def test_parallel_equals_whole(shape, mode, fos, bound):
    x = workloads.seeded_normal(*shape, seed=21, row_scale_decades=2.0)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    kw = dict(mode=mode, bound=bound, four_over_six=fos)
    _same(oracle.quantize_parallel(xb, "bf16", threads=3, strip=32, **kw),
          oracle.quantize(xb, "bf16", **kw))


@pytest.mark.parametrize("fos", [False, True])
def test_parallel_equals_whole_16x16_fp32(fos):
    x = workloads.seeded_normal(80, 112, seed=22, dtype=torch.float32).numpy()
    kw = dict(mode=oracle.PER_TENSOR, four_over_six=fos, block_2d=True)
    _same(oracle.quantize_parallel(x, "fp32", threads=4, strip=16, **kw),
          oracle.quantize(x, "fp32", **kw))


def test_parallel_one_direction():
    x = workloads.seeded_normal(70, 90, seed=23, dtype=torch.float32).numpy()
    for rw, cw in ((True, False), (False, True)):
        p = oracle.quantize_parallel(x, "fp32", rowwise=rw, columnwise=cw, threads=2, strip=16)
        w = oracle.quantize(x, "fp32", rowwise=rw, columnwise=cw)
        assert set(p) == set(w)
        _same(p, w)
