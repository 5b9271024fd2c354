"""The encode kernels' division by a decoded block scale on the GPU, against the
IEEE quotient.

The encode factor of a block, e = fl(S / sd) ("NVFP4: enable row-scaled transpose
quantization for backward", TransformerEngine PR #3206: the global and the block
scale of each line), is computed with a reciprocal and two FMA steps rather than a
division.  tests/test_kernel_division.py proves that this gives the correctly
rounded quotient when the reciprocal is itself correctly rounded; this test runs the
device routine for every E4M3 scale and many S, including the range edges where the
kernels switch to the IEEE division, and compares with numpy's float32 division
(correctly rounded).
"""
import numpy as np
import pytest
import torch

nv = pytest.importorskip("nvfp4_precision_quantization_gb300")

pytestmark = pytest.mark.gpu


def _e4m3_values():
    import oracle
    return np.array([oracle.lib().oracle_e4m3_decode(k) for k in range(127)], np.float32)


def test_scale_division_is_the_ieee_quotient():
    rng = np.random.default_rng(11)
    exps = rng.integers(-126, 101, 30000)
    man = rng.integers(0, 1 << 23, 30000)
    S = ((exps + 127).astype(np.uint32) << 23 | man.astype(np.uint32)).view(np.float32)
    edges = []
    for v in (2.0 ** -90, 2.0 ** 90, 1.0, 1536.0, 2688.0, 2688.0 / 448.0, 2.0 ** -126):
        b = int(np.array([v], np.float32).view(np.uint32)[0])
        edges.append(np.arange(b - 3, b + 4, dtype=np.uint32).view(np.float32))
    S = np.concatenate([S] + edges).astype(np.float32)
    S = S[np.isfinite(S) & (S > 0)]
    St = torch.from_numpy(S).cuda()
    e = torch.empty(S.size * 127, dtype=torch.float32, device="cuda")
    nv.nvfp4_selftest_scale_division(St, e)
    got = e.cpu().numpy().reshape(S.size, 127)
    sd = _e4m3_values()
    with np.errstate(divide="ignore", over="ignore"):
        want = np.where(sd[None, :] == 0, np.float32(0), S[:, None] / sd[None, :])
    bad = np.argwhere(got.view(np.uint32) != want.astype(np.float32).view(np.uint32))
    assert bad.size == 0, [(float(S[i]), int(k), float(got[i, k]), float(want[i, k]))
                           for i, k in bad[:5]]
