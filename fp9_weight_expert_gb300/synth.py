"""Seeded synthetic inputs for the fp9 FFN/MoE decode step.

This module only draws random numbers: it holds none of the method's
arithmetic (no encoding, routing or FFN math). Both the GPU path and the CPU
oracle receive the same fp32 tensors drawn here; each side then packs and
computes on its own.

Workload shapes (DeepSeek-V3-class MoE layer and its dense first layers):

  tiny   hidden 256, 8 routed experts of intermediate 128 in 1 group, top-2,
         route scale 1.0, 1 shared expert of intermediate 128;
         x ~ N(0,1), W_g ~ N(0, 0.05), expert weights ~ N(0, 0.02).
  dsv3   hidden 7168, 256 routed experts of intermediate 2048 in 8 groups of
         32, top-4 groups, top-8 experts, route scale 2.5, 1 shared expert;
         x ~ N(0,1), expert weights ~ N(0, 0.02), W_g ~ N(0, sigma_g) with
         sigma_g = 0.05 * sqrt(256 / 7168), which gives the router logits the
         same spread (std 0.8) as the tiny layer.
  dense  hidden 7168, one SwiGLU FFN of intermediate 18432,
         weights ~ N(0, 0.02), x ~ N(0,1).
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    hidden: int
    inter: int
    n_experts: int
    n_groups: int
    topk_groups: int
    topk: int
    n_shared: int
    route_scale: float
    router_std: float
    weight_std: float = 0.02


TINY = MoEShape(hidden=256, inter=128, n_experts=8, n_groups=1, topk_groups=1,
                topk=2, n_shared=1, route_scale=1.0, router_std=0.05)
DSV3 = MoEShape(hidden=7168, inter=2048, n_experts=256, n_groups=8,
                topk_groups=4, topk=8, n_shared=1, route_scale=2.5,
                router_std=0.05 * math.sqrt(256.0 / 7168.0))
DENSE_HIDDEN = 7168
DENSE_INTER = 18432

# Matrix indices inside one FFN.
GATE, UP, DOWN_T = 0, 1, 2
# Bank kinds.
ROUTED, SHARED, DENSE, ROUTER, TOKENS = 0, 1, 2, 3, 4


def seed_for(base: int, layer: int, kind: int, index: int = 0, matrix: int = 0) -> int:
    """A distinct 63-bit seed per (base, layer, kind, expert, matrix)."""
    v = (base & 0xFFFFFFFF)
    for part in (layer, kind, index, matrix):
        v = (v * 0x9E3779B97F4A7C15 + (part & 0xFFFFFFFF) + 1) & ((1 << 64) - 1)
        v ^= v >> 29
    return v & ((1 << 63) - 1)


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 tensor ~ N(0, std^2), drawn on ``device`` from ``seed``."""
    g = _generator(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def tokens(bsz: int, hidden: int, seed: int, device="cpu") -> torch.Tensor:
    """Token hidden states x [bsz, hidden] ~ N(0, 1)."""
    return normal((bsz, hidden), 1.0, seed, device)


def ffn_weight(shape: MoEShape | None, rows: int, cols: int, seed: int,
               device="cpu", std: float = 0.02) -> torch.Tensor:
    """One FFN matrix [rows, cols] ~ N(0, std^2) (gate, up or down_t)."""
    return normal((rows, cols), shape.weight_std if shape else std, seed, device)
