"""Four-over-six with both directions at sizes where every persistent CTA walks
several tiles, compared byte for byte with the oracle.

The encode kernel runs min(tiles, 2 x SMs) CTAs, each over a contiguous chunk of
the tile order, so the small parity shapes give every CTA one tile at most.  These
shapes give each CTA two to eight tiles.  That exercises the ring wrap, the tile
cursor's walk (the columnwise pass walks each chunk the other way) and the scale
stores with the four-over-six block choice ("Add NVFP4 four-over-six grouped GEMM
for MoE training", torchao PR #9, description: the block scaled to 4 or to 6 by the
lower squared error, bound 448 or 256) with both directions ("NVFP4: enable
row-scaled transpose quantization for backward", TransformerEngine PR #3206,
description).  With 1x16 blocks each direction is its own encode pass; the
shapes cover its output paths:

* 4096 x 4096 (the outliers workload): columnwise code pitch a multiple of 32
  bytes, one 32-byte sector store per lane pair; 1024 tiles.
* 3232 x 9184 and 4000 x 5000: pitches multiples of 16 but not of 32 bytes, or
  neither: direct 16-byte, 4-byte or byte stores; 936 and 640 tiles (BF16), 2528
  (4000 x 5000 FP32).  The rowwise pass stores directly on every shape.

The oracle runs in host threads over strips of lines (oracle.quantize_parallel, held
equal to the whole-tensor oracle by tests/test_oracle_parallel.py).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_helpers import assert_same, cfg, gpu_quantize, host_bits

nv = pytest.importorskip("nvfp4_precision_quantization_gb300")

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = {
    "sector_4096x4096": lambda: workloads.outliers(DEV),
    "direct_3232x9184": lambda: workloads.seeded_normal(3232, 9184, seed=31, device=DEV,
                                                        row_scale_decades=2.0),
    "direct_4000x5000_bf16": lambda: workloads.edge_normal(4000, 5000, torch.bfloat16, DEV),
    "direct_4000x5000_fp32": lambda: workloads.edge_normal(4000, 5000, torch.float32, DEV),
}


def _output_path(rows, cols, dtype):
    """The columnwise pass's store path for these pitches (the rowwise pass of
    four-over-six stores directly): whole sectors when the BF16 code pitch is a
    multiple of 32 bytes."""
    if dtype != torch.bfloat16:
        return "direct"
    return "sector" if ((rows + 1) // 2) % 32 == 0 else "direct"


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    x = CASES[request.param]()
    return request.param, x, host_bits(x)


@pytest.mark.parametrize("mode", [nv.NVFP4_ROW_SCALED, nv.NVFP4_PER_TENSOR])
@pytest.mark.parametrize("bound", [256.0, 448.0])
def test_fos_both_directions_multitile_full(case, mode, bound):
    name, x, (xb, tag) = case
    rows, cols = x.shape
    assert name.startswith(_output_path(rows, cols, x.dtype))
    tiles = -(-rows // 128) * -(-cols // (128 if x.dtype == torch.bfloat16 else 64))
    assert tiles > 2 * 152  # more tiles than CTAs: the chunks hold several tiles
    c = cfg(mode, bound, fos=True)
    g = gpu_quantize(x, c)
    o = oracle.quantize_parallel(xb, tag, mode=mode, bound=bound, four_over_six=True)
    assert_same(g["row"], o["row"], f"{name} row")
    assert_same(g["col"], o["col"], f"{name} col")


def test_fos_choice_is_exercised(case):
    """The inputs make both candidates win somewhere (else the test above could not
    tell a kernel that ignores the T = 4 candidate from a correct one)."""
    name, x, (xb, tag) = case
    n = min(512, x.shape[0])
    part = xb[:n]
    on = oracle.quantize(part, tag, mode=oracle.ROW_SCALED, bound=256.0, four_over_six=True,
                         columnwise=False)["row"]
    off = oracle.quantize(part, tag, mode=oracle.ROW_SCALED, bound=256.0, four_over_six=False,
                          columnwise=False)["row"]
    changed = (on[1] != off[1]).mean()
    assert 0.05 < changed < 0.95, (name, changed)
