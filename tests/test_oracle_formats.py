"""Pins for the oracle's number formats (CPU only).

Each conversion in the oracle is checked against an independent formulation:
  * E2M1 encode  vs  "divide by the binade spacing, round half to even with
    numpy.rint, clamp at 6" computed in float64;
  * E2M1 decode  vs  the closed form (-1)^s * (e == 0 ? m/2 : (1 + m/2) 2^(e-1));
  * E4M3 encode  vs  torch's float8_e4m3fn conversion (RNE) below 464, and vs the
    same spacing formulation as E2M1; saturation to 448 checked separately;
  * E4M3 decode  vs  torch's float8_e4m3fn -> float32 for all 256 codes;
  * BF16         vs  torch's bfloat16 conversions.
"""
import numpy as np
import pytest
import torch

import oracle

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _neighbours(values, radius):
    """All finite float32 within +-radius ulps of each positive value, and their negations."""
    out = []
    for v in values:
        b = int(np.array([v], np.float32).view(np.int32)[0])
        k = np.arange(b - radius, b + radius + 1, dtype=np.int64)
        k = k[(k >= 0) & (k < 0x7F800000)]
        out.append(k.astype(np.uint32).view(np.float32))
    f = np.concatenate(out)
    return np.concatenate([f, -f])


def _all_bf16_as_f32():
    h = np.arange(65536, dtype=np.uint32) << 16
    f = h.view(np.float32)
    return f[~np.isnan(f)]


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    logu = rng.uniform(np.log(1e-4), np.log(1e3), size=n)
    g = (np.exp(logu) * rng.choice([-1.0, 1.0], size=n)).astype(np.float32)
    return np.concatenate([f, g])


def e2m1_reference(y: np.ndarray) -> np.ndarray:
    y = y.astype(np.float32)
    m = np.abs(y.astype(np.float64))
    spacing = np.where(m < 2.0, 0.5, np.where(m < 4.0, 1.0, 2.0))
    q = np.minimum(np.rint(m / spacing) * spacing, 6.0)
    code = np.searchsorted(E2M1_VALUES, q).astype(np.uint8)
    assert np.all(E2M1_VALUES[code] == q)
    return code | (np.signbit(y).astype(np.uint8) << 3)


def e4m3_reference_spacing(s: np.ndarray) -> np.ndarray:
    """RNE onto the E4M3 grid via binade spacing, saturating at 448; magnitude code."""
    m = np.minimum(np.abs(s.astype(np.float64)), 1e30)  # beyond 448 everything saturates
    safe = np.maximum(m, 2.0**-6)
    exp = np.floor(np.log2(safe))
    # log2 can be off by one near powers of two: correct it exactly
    exp = np.where(2.0**exp > safe, exp - 1, exp)
    exp = np.where(2.0**(exp + 1) <= safe, exp + 1, exp)
    spacing = np.where(m < 2.0**-6, 2.0**-9, 2.0**(exp - 3))
    q = np.minimum(np.rint(m / spacing) * spacing, 448.0)
    grid = np.array([oracle.lib().oracle_e4m3_decode(k) for k in range(0x7F)], np.float64)
    code = np.searchsorted(grid, q)
    assert np.all(grid[code] == q)
    return code.astype(np.uint8) | (np.signbit(s).astype(np.uint8) << 7)


def _e2m1_inputs():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0]
    pts = list(E2M1_VALUES[1:]) + mids + [8.0, 12.0]
    return np.concatenate([_all_bf16_as_f32(), _neighbours(pts, 3000),
                           _neighbours([2.0**-126, 2.0**-149 * 3], 50),
                           _random_f32(1_000_000, 7),
                           np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45], np.float32)])


def test_e2m1_encode_matches_spacing_rule():
    y = _e2m1_inputs()
    got = oracle.e2m1_encode(y)
    ref = e2m1_reference(y)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (y[bad[:10]], got[bad[:10]], ref[bad[:10]])


@pytest.mark.parametrize("y,code", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4),
                                    (3.5, 6), (5.0, 6), (6.0, 7), (7.0, 7), (1e30, 7),
                                    (-0.25, 8), (-0.0, 8), (0.0, 0), (-1e-30, 8), (-5.0, 14),
                                    (0.2500001, 1), (0.7499999, 1)])
def test_e2m1_ties_and_signs(y, code):
    assert int(oracle.e2m1_encode(np.array([y], np.float32))[0]) == code


def test_e2m1_decode_closed_form():
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        want = -mag if s else mag
        got = float(oracle.e2m1_decode(np.array([c], np.uint8))[0])
        assert got == want and np.signbit(got) == bool(s)


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = oracle.e4m3_decode(codes.numpy())
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert oracle.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0**-9
    assert oracle.e4m3_decode(np.array([0x38], np.uint8))[0] == 1.0


def _e4m3_inputs():
    grid = np.array([oracle.lib().oracle_e4m3_decode(k) for k in range(0x7F)], np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([grid[1:], mids]).astype(np.float32)
    return np.concatenate([_all_bf16_as_f32(), _neighbours(pts, 40), _random_f32(300_000, 11)])


def test_e4m3_encode_matches_torch_below_464():
    s = _e4m3_inputs()
    s = s[np.abs(s) < 464.0]
    got = oracle.e4m3_encode(s)
    ref = torch.from_numpy(s.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (s[bad[:10]], got[bad[:10]], ref[bad[:10]])


def test_e4m3_encode_matches_spacing_rule_and_saturates():
    s = _e4m3_inputs()
    got = oracle.e4m3_encode(s)
    ref = e4m3_reference_spacing(s)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (s[bad[:10]], got[bad[:10]], ref[bad[:10]])
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    # below half the smallest subnormal -> 0; the tie at exactly 2^-10 goes to even (0)
    tiny = np.array([2.0**-11, 2.0**-10, np.nextafter(np.float32(2.0**-10), np.float32(1))],
                    np.float32)
    assert list(oracle.e4m3_encode(tiny)) == [0, 0, 1]


def test_bf16_conversions_match_torch():
    h = np.arange(65536, dtype=np.uint16)
    f = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(f.view(np.uint32), ref.view(np.uint32)) or np.all(
        (f == ref) | (np.isnan(f) & np.isnan(ref)))
    x = _random_f32(200_000, 3)
    got = oracle.f32_to_bf16(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_no_fused_multiply_add():
    # (1+2^-12)^2 - (1+2^-11) is 0 with two roundings and 2^-24 with an FMA.
    a = 1.0 + 2.0**-12
    assert oracle.lib().oracle_fp_contract_probe(a, a, -(1.0 + 2.0**-11)) == 0.0
