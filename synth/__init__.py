"""Seeded synthetic inputs shared by the tests, the smoke entry and the bench.

This module holds no arithmetic of the method: it only draws bf16 tensors of
the shapes and value distributions of the workloads (the pages' draft layers
cannot be loaded here; there are no trained weights).  The recipe:

  * generator ``torch.Generator('cpu').manual_seed(seed)``;
  * ``randn`` in fp32, multiplied by ``sigma``;
  * optional per-row scale ``exp(U[ln lo, ln hi])`` (log-uniform), applied
    before the outliers;
  * outliers: exactly ``round(frac * numel)`` positions drawn by ``randperm``
    (same generator), multiplied by ``mult``;
  * finally one cast to bf16 (round to nearest even).

Shapes come from the pages: the o_proj weight (7168, 8192) of "Exact
quantization coverage" ("Kimi-K3 DSpark O-Proj-only MXFP4"), M = 8 tokens per
request (1 verified + 7 drafted, 7 speculative tokens) and concurrency 8 from
the performance-test sentence under "Why O-proj only", 1024-token prompts.
The FP8 MLP width 18432 is synthetic (the pages do not state it).
"""
from __future__ import annotations

import math

import torch

# o_proj shape (out_features N, in_features K) of the stored MXFP4 weight
OPROJ_N, OPROJ_K = 7168, 8192
# synthetic MLP intermediate width for the FP8 gate_up / down pair
MLP_I = 18432


def bf16_randn(rows: int, cols: int, seed: int, sigma: float = 1.0,
               outlier_frac: float = 0.0, outlier_mult: float = 50.0,
               row_scale_range: tuple[float, float] | None = None) -> torch.Tensor:
    """(rows, cols) bf16 CPU tensor drawn per the recipe above."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    if row_scale_range is not None:
        lo, hi = row_scale_range
        u = torch.rand(rows, 1, generator=g, dtype=torch.float32)
        x.mul_(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    n_out = int(round(outlier_frac * rows * cols))
    if n_out > 0:
        pos = torch.randperm(rows * cols, generator=g)[:n_out]
        x.view(-1)[pos] *= outlier_mult
    return x.to(torch.bfloat16)


def weight(n: int, k: int, seed: int) -> torch.Tensor:
    """Weight matrix W (n, k): bf16 N(0, 0.02), no outliers."""
    return bf16_randn(n, k, seed, sigma=0.02)


def activation(m: int, k: int, seed: int, row_scale: bool = False) -> torch.Tensor:
    """Activation X (m, k): bf16 N(0, 1) with 0.1% of entries x50; optional
    log-uniform per-row scale in [0.1, 10] (the prefill workload)."""
    return bf16_randn(m, k, seed, sigma=1.0, outlier_frac=0.001, outlier_mult=50.0,
                      row_scale_range=(0.1, 10.0) if row_scale else None)


def act_seed(cfg: int, layer: int, gemm_idx: int) -> int:
    """Activation seed of (workload, layer, GEMM index)."""
    return 1000 + 100 * cfg + 10 * layer + gemm_idx


# Weight seeds per workload.
SEED_CFG0_W = 0                      # single o_proj layer, M = 8
SEEDS_CFG1_W = (1, 2, 3, 4, 5)       # 5-layer o_proj decode chain, M = 64
SEED_CFG2_W = 6                      # o_proj prefill, M = 8192
SEED_CFG3_GATE_UP, SEED_CFG3_DOWN = 7, 8  # FP8 MLP pair


def seed_cfg4(kind: str, layer: int) -> int:
    """Mixed-precision sweep weights: o_proj 20+l, gate_up 30+l, down 40+l."""
    return {"o_proj": 20, "gate_up": 30, "down": 40}[kind] + layer


# MLA up-projections of the draft layer, FP8 PTPC (the pages list q_b_proj
# and kv_b_proj among the FP8 weights but give no shapes; synthetic, from the
# usual MLA layout with 64 heads): (N, K) = (64 x (128 + 64), 1536) and
# (64 x (128 + 128), 512); weight seeds 70 and 71.
MLA_QB, MLA_KVB = (12288, 1536), (16384, 512)
SEED_MLA_QB, SEED_MLA_KVB = 70, 71

# Synthetic expert layer (the pages give no expert shapes): gate_up of a
# 2048-wide expert over the 7168-wide hidden state, 8 experts, 8192 routed
# token rows (e.g. 1024 tokens x top-8), seed 60 + e for expert e's weight.
MOE_EXPERTS, MOE_N, MOE_K, MOE_ROWS = 8, 4096, 7168, 8192
SEED_MOE_W, SEED_MOE_ROUTE = 60, 61


def group_sizes(rows: int, groups: int, seed: int) -> list:
    """Uneven seeded group sizes summing to `rows`: each row goes to a group
    drawn from a seeded Dirichlet(3)-weighted categorical distribution."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    # Dirichlet(3) weights from the generator: normalised sums of 3 exponentials
    e = -torch.log(torch.rand(groups, 3, generator=g, dtype=torch.float64)).sum(dim=1)
    p = e / e.sum()
    pick = torch.multinomial(p, rows, replacement=True, generator=g)
    return torch.bincount(pick, minlength=groups).tolist()


def special_values_bf16() -> torch.Tensor:
    """A row of edge-case bf16 bit patterns for quantizer edge tests: +-0,
    the smallest/largest subnormals and normals, the E2M1 rounding midpoints
    at unit scale, and huge magnitudes (no NaN/Inf)."""
    bits = [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F,
            0x3E80, 0x3F40, 0x3FA0, 0x3FE0, 0x4020, 0x4060, 0x40A0, 0xBE80,
            0xBF40, 0xBFA0, 0xBFE0, 0xC020, 0xC060, 0xC0A0, 0x3F80, 0xBF80,
            0x40C0, 0xC0C0, 0x4100, 0x3DCC, 0xBDCC, 0x0040, 0x8040, 0x3C00]
    return torch.tensor(bits, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
