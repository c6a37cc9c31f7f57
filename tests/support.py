"""Helpers shared by the GPU parity tests and smoke(): build fp9 layers on
the GPU from the seeded generators, and build the oracle's inputs from the
same fp32 draws (the oracle packs them itself; nothing it sees comes from
the CUDA path)."""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
from fp9_weight_expert_gb300 import layers, synth

MARGIN_MIN = 1e-4   # routing decisions closer than this are redrawn
TOL = 2e-4          # max|gpu - oracle| <= TOL * max|oracle| per output vector


def ffn_source(shape: synth.MoEShape, base: int, layer: int, bank: int, k: int, m: int, device):
    kind = synth.ROUTED if bank == 0 else synth.SHARED
    return synth.ffn_weight(shape, shape.inter, shape.hidden,
                            synth.seed_for(base, layer, kind, k, m), device)


def router_source(shape: synth.MoEShape, base: int, layer: int, device):
    return synth.normal((shape.n_experts, shape.hidden), shape.router_std,
                        synth.seed_for(base, layer, synth.ROUTER), device)


def build_layer(shape: synth.MoEShape, base: int = 1, layer: int = 0, device="cuda",
                status: torch.Tensor | None = None) -> layers.MoELayer:
    L = layers.MoELayer(shape.hidden, shape.inter, shape.n_experts, shape.n_groups,
                        shape.topk_groups, shape.topk, shape.n_shared, shape.route_scale, device)
    L.fill(lambda b, k, m: ffn_source(shape, base, layer, b, k, m, device),
           router_source(shape, base, layer, device), status)
    return L


class OracleLayer:
    """Oracle view of a layer: packs each expert's fp32 draw with the
    oracle's own encoder, on demand."""

    def __init__(self, shape: synth.MoEShape, base: int = 1, layer: int = 0, device="cuda"):
        self.shape, self.base, self.layer, self.device = shape, base, layer, device
        self.w_router = router_source(shape, base, layer, device).cpu().numpy()
        self._cache = {}

    def planes(self, bank: int, k: int):
        key = (bank, k)
        if key not in self._cache:
            out = []
            for m in range(3):
                w = ffn_source(self.shape, self.base, self.layer, bank, k, m, self.device)
                body, sign, err = O.fp9_pack(w.cpu().numpy())
                assert not err
                out += [body, sign]
            self._cache[key] = tuple(out)
        return self._cache[key]

    def kwargs(self):
        s = self.shape
        return dict(w_router=self.w_router, routed=lambda e: self.planes(0, e),
                    shared=[self.planes(1, k) for k in range(s.n_shared)],
                    n_groups=s.n_groups, topk_groups=s.topk_groups, topk=s.topk,
                    route_scale=s.route_scale)

    def route(self, x):
        s = self.shape
        return O.route(x, self.w_router, s.n_groups, s.topk_groups, s.topk, s.route_scale)

    def margin(self, x):
        s = self.shape
        return O.route_margin(x, self.w_router, s.n_groups, s.topk_groups, s.topk)


def safe_tokens(shape: synth.MoEShape, w_router: np.ndarray, bsz: int, base: int, layer: int = 0,
                device="cpu") -> torch.Tensor:
    """bsz token rows ~ N(0,1), each redrawn (next seed) until every routing
    decision has a margin of at least MARGIN_MIN in the oracle's float64."""
    rows = []
    for t in range(bsz):
        for attempt in range(1000):
            x = synth.tokens(1, shape.hidden, synth.seed_for(base, layer, synth.TOKENS, t, attempt), "cpu")
            m = O.route_margin(x.numpy(), w_router, shape.n_groups, shape.topk_groups, shape.topk)
            if m[0] >= MARGIN_MIN:
                rows.append(x)
                break
        else:  # pragma: no cover
            raise RuntimeError("no token with a safe routing margin")
    return torch.cat(rows).to(device)


def max_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of max|gpu - ref| / max|ref| (the per-vector rule)."""
    gpu = np.atleast_2d(gpu).astype(np.float64)
    ref = np.atleast_2d(ref).astype(np.float64)
    out = 0.0
    for g, r in zip(gpu, ref):
        out = max(out, float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30)))
    return out
