"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays out tensors; it holds none of
the NVFP4 arithmetic.  The CUDA path and the CPU oracle both consume what it
returns (the oracle through a host copy of the very same bytes).

Workloads (the pages quote no dataset; these stand in for the training
operands they describe):
  tiny        256 x 256 BF16, N(0,1) times a per-row factor log-uniform in
              [1e-2, 1e2] (seed 0): row-scaled both directions, bound 448.
  outliers    4096 x 4096 BF16, N(0,1) with 0.1 % of the entries (chosen
              uniformly without replacement) multiplied by 50 (seed 1).
  linear      activation X 16384 x 8192 and gradient dY 16384 x 28672 BF16,
              N(0, 0.02) times a per-row LogNormal(0, 1) magnitude (seed 2).
  moe         32 expert groups, token counts Multinomial(65536, uniform) (seed 3),
              each group zero-padded to a multiple of 128 rows, K = 7168, N(0,1).
  edge        4000 x 5000 N(0,1) in BF16 and FP32, 8192 x 8192 N(0, 0.02),
              4096 x 4096 with every 8th row zero, an all-zero tensor (seed 4).
  moe-gemm    the grouped GEMM of the MoE layout above: the padded tokens' NVFP4 bytes
              (K 7168) times 32 experts' weights (N 2048), drawn like `gemm` below,
              one per-tensor amax per expert (seed 5 and up).
  gemm        NVFP4 operand bytes for the GEMM consumer, drawn directly: code bytes
              uniform over all 256 values (every pair of E2M1 codes, both signs),
              scale bytes uniform over the normal positive E4M3 codes 0x08..0x7E,
              amax log-uniform in [1e-2, 1e2] per line (or one value per tensor).
              Shapes of the linear layer above: fprop X (16384 x 8192) times the
              weight W (28672 x 8192)^T, wgrad dY^T (28672 x 16384) times X^T
              (8192 x 16384)^T (seed 5 and up).
"""
from __future__ import annotations

import math

import torch

SEEDS = {"tiny": 0, "outliers": 1, "linear": 2, "moe": 3, "edge": 4, "gemm": 5}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def tiny(device="cpu") -> torch.Tensor:
    g = generator(SEEDS["tiny"], device)
    x = torch.randn(256, 256, generator=g, device=device)
    u = torch.rand(256, 1, generator=g, device=device)
    lo, hi = math.log(1e-2), math.log(1e2)
    return (x * torch.exp(lo + (hi - lo) * u)).to(torch.bfloat16)


def outliers(device="cpu", rows: int = 4096, cols: int = 4096) -> torch.Tensor:
    g = generator(SEEDS["outliers"], device)
    x = torch.randn(rows, cols, generator=g, device=device)
    n_out = round(0.001 * rows * cols)
    idx = torch.randperm(rows * cols, generator=g, device=device)[:n_out]
    x.view(-1)[idx] *= 50.0
    return x.to(torch.bfloat16)


def row_lognormal(rows: int, cols: int, g: torch.Generator, device, std: float = 0.02,
                  chunk_rows: int = 2048) -> torch.Tensor:
    """N(0, std) times a per-row LogNormal(0, 1) factor, built in row chunks so the
    FP32 temporaries stay small."""
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn(r1 - r0, cols, generator=g, device=device) * std
        f = torch.exp(torch.randn(r1 - r0, 1, generator=g, device=device))
        out[r0:r1] = (x * f).to(torch.bfloat16)
    return out


def linear(device="cpu", rows: int = 16384, k_x: int = 8192, k_dy: int = 28672):
    """(X, dY) linear-layer operands."""
    g = generator(SEEDS["linear"], device)
    x = row_lognormal(rows, k_x, g, device)
    dy = row_lognormal(rows, k_dy, g, device)
    return x, dy


def moe_counts(num_groups: int = 32, tokens: int = 65536, device="cpu") -> torch.Tensor:
    g = generator(SEEDS["moe"], "cpu")
    draws = torch.randint(0, num_groups, (tokens,), generator=g)
    return torch.bincount(draws, minlength=num_groups).to(torch.int64)


def moe_layout(num_groups: int = 32, tokens: int = 65536, align: int = 128):
    """The MoE token counts, their padded counts and the padded group ends (CPU int64),
    without generating any tokens."""
    counts = moe_counts(num_groups, tokens)
    padded = ((counts + align - 1) // align) * align
    return counts, padded, torch.cumsum(padded, 0)


def moe(device="cpu", num_groups: int = 32, tokens: int = 65536, cols: int = 7168,
        align: int = 128):
    """Ragged token groups zero-padded to ``align`` rows.

    Returns (x_padded [M_pad, cols] bf16, group_ends [G] int64 on ``device``,
    counts [G] int64 (unpadded, CPU), padded_counts [G] int64 (CPU)).
    Real rows are N(0,1); padding rows are +0.
    """
    counts = moe_counts(num_groups, tokens)
    padded = ((counts + align - 1) // align) * align
    ends = torch.cumsum(padded, 0)
    m_pad = int(ends[-1])
    g = generator(SEEDS["moe"] + 1000, device)
    x = torch.zeros(m_pad, cols, dtype=torch.bfloat16, device=device)
    start = 0
    for c, p in zip(counts.tolist(), padded.tolist()):
        if c:
            x[start:start + c] = torch.randn(c, cols, generator=g, device=device).to(torch.bfloat16)
        start += p
    return x, ends.to(device), counts, padded


def moe_ragged(x_padded: torch.Tensor, counts: torch.Tensor, padded: torch.Tensor):
    """The unpadded token tensor and its group ends, sliced out of the padded one."""
    parts, start = [], 0
    for c, p in zip(counts.tolist(), padded.tolist()):
        parts.append(x_padded[start:start + c])
        start += p
    return torch.cat(parts, 0), torch.cumsum(counts, 0)


def edge_normal(rows: int = 4000, cols: int = 5000, dtype=torch.bfloat16, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    g = generator(SEEDS["edge"], device)
    return (torch.randn(rows, cols, generator=g, device=device) * std).to(dtype)


def edge_zero_rows(rows: int = 4096, cols: int = 4096, every: int = 8, device="cpu"):
    g = generator(SEEDS["edge"] + 1, device)
    x = torch.randn(rows, cols, generator=g, device=device)
    x[::every] = 0.0
    return x.to(torch.bfloat16)


def seeded_normal(rows: int, cols: int, seed: int, dtype=torch.bfloat16, device="cpu",
                  std: float = 1.0, row_scale_decades: float = 0.0) -> torch.Tensor:
    """General N(0, std) input for parity sweeps; optional per-row log-uniform
    factor spanning +-row_scale_decades decades."""
    g = generator(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device) * std
    if row_scale_decades:
        u = torch.rand(rows, 1, generator=g, device=device) * 2.0 - 1.0
        x = x * torch.pow(10.0, row_scale_decades * u)
    return x.to(dtype)


def nvfp4_operand(lines: int, k: int, seed: int, row_scaled: bool = True, device="cpu"):
    """Random NVFP4 operand bytes (codes [lines][k/2], scales [lines][k/16], amax
    [lines] or [1]) for the GEMM consumer; see the module docstring."""
    g = generator(SEEDS["gemm"] * 1000 + seed, device)
    codes = torch.randint(0, 256, (lines, k // 2), generator=g, device=device, dtype=torch.int32)
    scales = torch.randint(0x08, 0x7F, (lines, k // 16), generator=g, device=device,
                           dtype=torch.int32)
    u = torch.rand(lines if row_scaled else 1, generator=g, device=device)
    lo, hi = math.log(1e-2), math.log(1e2)
    amax = torch.exp(lo + (hi - lo) * u).to(torch.float32)
    return codes.to(torch.uint8), scales.to(torch.uint8), amax


# linear-layer GEMM shapes (m, n, k): fprop Y = X W^T and wgrad dW = dY^T X
GEMM_SHAPES = {"fprop": (16384, 28672, 8192), "wgrad": (28672, 8192, 16384)}
