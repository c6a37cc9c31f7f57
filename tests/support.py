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


# ---------------------------------------------------------------- prefill ---
# fp9_ffn_prefill rounds x and h = SiLU(g) * u to fp16 (the tensor cores'
# operand type; the fp9 weights are exact in fp16) and accumulates in fp32.
# Its tolerance against the exact FFN comes from that arithmetic:
#   * element-wise, a worst-case first-order bound (prefill_error_bound);
#   * in aggregate, the relative L2 error of two independent fp16 roundings
#     of the GEMM operands: each contributes about u16 / sqrt(3) = 2.8e-4
#     relative, together about 3.7e-4 (measured on an fp16 emulation of the
#     path at three shapes). The limits below leave 1.6x (global) and 2.3x
#     (per row) headroom, and reject rounding h to bf16 (1.7e-3) or dropping
#     one 64-wide K chunk (>= 0.08).
PREFILL_FRO = 6e-4    # ||y - y_exact||_F / ||y_exact||_F over a whole output
PREFILL_ROW = 1.2e-3  # the same for each token row
U16 = 2.0 ** -11      # unit roundoff of fp16, round to nearest even
F16_SUB = 2.0 ** -25  # half the spacing of fp16 subnormals


def prefill_error_bound(x, wg, wu, wd):
    """Worst-case |y_path - y_exact| per element for the fp16-operand path.

    x [m, H] (fp64), wg/wu [I, H] and wd = down_t [I, H] decoded weights.
    Terms: fp16 rounding of x (relative U16, or F16_SUB absolute for
    subnormals); fp32 accumulation of K exact products, allowing one ulp per
    addition (gamma = K * 2^-23); |SiLU'| <= 1.1; a few fp32 ulps for the
    SiLU and the product; fp16 rounding of h; then the same accumulation
    bound for the down GEMM over I terms.
    """
    x = np.asarray(x, np.float64)
    K, I = x.shape[1], wg.shape[0]
    gk, gi = K * 2.0 ** -23, I * 2.0 ** -23
    ax = np.abs(x)
    awg, awu, awd = np.abs(wg), np.abs(wu), np.abs(wd)
    g, u = x @ wg.T, x @ wu.T
    dg = (U16 + gk * (1 + U16)) * (ax @ awg.T) + F16_SUB * awg.sum(1) * (1 + gk)
    du = (U16 + gk * (1 + U16)) * (ax @ awu.T) + F16_SUB * awu.sum(1) * (1 + gk)
    s = g / (1.0 + np.exp(-g))
    h = s * u
    dh0 = 1.1 * dg * (np.abs(u) + du) + np.abs(s) * du + 4 * 2.0 ** -24 * np.abs(h)
    dh = dh0 + U16 * (np.abs(h) + dh0) + F16_SUB
    return dh @ awd + gi * ((np.abs(h) + dh) @ awd)


def prefill_errors(y, y_exact):
    """(global relative L2 error, largest per-row relative L2 error)."""
    y = np.asarray(y, np.float64)
    y_exact = np.asarray(y_exact, np.float64)
    d = y - y_exact
    fro = float(np.linalg.norm(d) / max(np.linalg.norm(y_exact), 1e-300))
    rows = np.linalg.norm(d, axis=1) / np.maximum(np.linalg.norm(y_exact, axis=1), 1e-300)
    return fro, float(rows.max())


def check_prefill(y, x, wg, wu, wd, y_exact=None):
    """Asserts the prefill tolerance for y [m, H] given the exact inputs."""
    if y_exact is None:
        y_exact = O.ffn(x, wg, wu, wd)
    bound = prefill_error_bound(x, wg, wu, wd)
    over = np.abs(np.asarray(y, np.float64) - y_exact) - bound
    assert over.max() <= 0.0, f"element-wise bound exceeded by {over.max():.3e}"
    fro, row = prefill_errors(y, y_exact)
    assert fro <= PREFILL_FRO, f"relative L2 error {fro:.3e} > {PREFILL_FRO}"
    assert row <= PREFILL_ROW, f"per-row relative L2 error {row:.3e} > {PREFILL_ROW}"
    return fro, row


def decoded(planes):
    """(W_gate, W_up, down_t) as float64 from an FFN's six packed planes."""
    return tuple(O.fp9_decode(planes[2 * i], planes[2 * i + 1]) for i in range(3))


def moe_prefill_bound(x, ol, ids, wts):
    """Element-wise bound for fp9_moe_prefill: each expert term's
    prefill_error_bound times |its routing weight| (1 for shared experts),
    plus fp32 rounding of the weighted sum (one ulp of the summed
    magnitudes per term)."""
    x = np.asarray(x, np.float64)
    m, topk = ids.shape
    bound = np.zeros_like(x)
    mag = np.zeros_like(x)
    for e in np.unique(ids):
        ts, ks = np.nonzero(ids == e)
        wg, wu, wd = decoded(ol.planes(0, int(e)))
        b = prefill_error_bound(x[ts], wg, wu, wd)
        y = O.ffn(x[ts], wg, wu, wd)
        w = np.abs(wts[ts, ks])[:, None]
        np.add.at(bound, ts, w * b)
        np.add.at(mag, ts, w * np.abs(y))
    for s in range(ol.shape.n_shared):
        wg, wu, wd = decoded(ol.planes(1, s))
        bound += prefill_error_bound(x, wg, wu, wd)
        mag += np.abs(O.ffn(x, wg, wu, wd))
    return bound + (topk + ol.shape.n_shared) * 2.0 ** -23 * mag


def check_moe_prefill(y, x, ol, ids, wts, y_exact):
    """Asserts the prefill tolerance (element-wise bound, relative L2) for
    an MoE layer's output y [m, H]."""
    bound = moe_prefill_bound(x, ol, ids, wts)
    over = np.abs(np.asarray(y, np.float64) - y_exact) - bound
    assert over.max() <= 0.0, f"element-wise bound exceeded by {over.max():.3e}"
    fro, row = prefill_errors(y, y_exact)
    assert fro <= PREFILL_FRO, f"relative L2 error {fro:.3e} > {PREFILL_FRO}"
    assert row <= PREFILL_ROW, f"per-row relative L2 error {row:.3e} > {PREFILL_ROW}"
    return fro, row
