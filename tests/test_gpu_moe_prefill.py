"""GPU parity for fp9_moe_prefill (an MoE layer over many tokens at once,
expert FFNs as grouped GEMMs on the tensor cores) against the oracle:
routing bit-exact on margin-safe tokens; outputs of the default precision
(activations as two fp16 terms) within the decode rule max|gpu - oracle|
<= 2e-4 * max|oracle| per token, those of the opt-in one-term fp16 mode
within its tolerance (support.check_moe_prefill)."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu

# 64 experts in 8 groups, 2 shared experts, top-6 of the best 4 groups
MID = synth.MoEShape(hidden=512, inter=128, n_experts=64, n_groups=8, topk_groups=4, topk=6, n_shared=2,
                     route_scale=2.5, router_std=0.05 * (64 / 512) ** 0.5)
# few experts with many tokens each (several token tiles per expert), no shared expert
FEW = synth.MoEShape(hidden=256, inter=256, n_experts=4, n_groups=1, topk_groups=1, topk=2, n_shared=0,
                     route_scale=1.0, router_std=0.05)
SHAPES = {"tiny": synth.TINY, "mid": MID, "few": FEW}


SPLIT, FP16 = binding.FP9_PREFILL_SPLIT, binding.FP9_PREFILL_FP16
PRECISIONS = pytest.mark.parametrize("precision", [SPLIT, FP16], ids=["split", "fp16"])


def _run(layer, x, status=None, precision=SPLIT):
    m = x.shape[0]
    y = torch.empty_like(x)
    ids = torch.empty((m, layer.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((m, layer.topk), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    binding.fp9_moe_prefill(layer, x, y, Workspace.for_moe_prefill(layer, m).tensor, st, ids, w,
                            precision=precision)
    torch.cuda.synchronize()
    return y, ids, w, int(st.item())


# few: 700 tokens over 4 experts, so each expert has several token tiles
# (128 rows each; 64-token halves in the gate/up GEMM of the default mode)
@pytest.mark.parametrize("name,m", [("tiny", 1), ("tiny", 37), ("tiny", 300), ("mid", 200), ("mid", 1000),
                                    ("few", 700)])
@PRECISIONS
def test_moe_prefill_matches_oracle(name, m, precision):
    shape = SHAPES[name]
    layer = support.build_layer(shape, base=31)
    ol = support.OracleLayer(shape, base=31)
    x = support.safe_tokens(shape, ol.w_router, m, base=m)
    y, ids, w, st = _run(layer, x.cuda(), precision=precision)
    assert st == 0
    xr = x.numpy().astype(np.float64)
    rid, rw = ol.route(xr)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(w.cpu().numpy() - rw).max() <= 1e-5 * shape.route_scale
    ref = O.moe(xr, **ol.kwargs())
    if precision == SPLIT:
        err = support.max_rel_err(y.cpu().numpy(), ref)
        assert err <= support.TOL, err
    else:
        support.check_moe_prefill(y.cpu().numpy(), xr, ol, rid, rw, ref)


def test_moe_prefill_agrees_with_the_decode_step():
    """The same tokens through fp9_moe_forward (8 at a time, fp32
    activations) give the same routing and outputs within the tolerance."""
    shape = MID
    layer = support.build_layer(shape, base=5)
    ol = support.OracleLayer(shape, base=5)
    x = support.safe_tokens(shape, ol.w_router, 64, base=3).cuda()
    y, ids, w, st = _run(layer, x)
    assert st == 0
    y16, ids16, _, st = _run(layer, x, precision=FP16)
    assert st == 0 and torch.equal(ids16, ids)
    yd = torch.empty_like(x)
    idd = torch.empty_like(ids)
    wd = torch.empty_like(w)
    ws = Workspace.for_moe(layer, 8).tensor
    for i in range(0, 64, 8):
        binding.fp9_moe_forward(layer, x[i:i + 8], yd[i:i + 8], ws, None, idd[i:i + 8], wd[i:i + 8])
    torch.cuda.synchronize()
    assert torch.equal(ids, idd)
    assert (w - wd).abs().max().item() <= 1e-6 * shape.route_scale
    assert support.max_rel_err(y.cpu().numpy(), yd.cpu().numpy()) <= support.TOL
    fro, row = support.prefill_errors(y16.cpu().numpy(), yd.cpu().numpy())
    assert fro <= support.PREFILL_FRO and row <= support.PREFILL_ROW


@PRECISIONS
def test_moe_prefill_is_deterministic(precision):
    layer = support.build_layer(MID, base=6)
    x = synth.tokens(500, MID.hidden, 77, "cuda")
    y1, i1, _, _ = _run(layer, x, precision=precision)
    y2, i2, _, _ = _run(layer, x, precision=precision)
    assert torch.equal(i1, i2) and torch.equal(y1, y2)


@PRECISIONS
def test_moe_prefill_flags_out_of_range_tokens(precision):
    layer = support.build_layer(synth.TINY, base=8)
    x = synth.tokens(20, synth.TINY.hidden, 9, "cuda")
    x[4, 3] = 1.0e5
    _, _, _, st = _run(layer, x, precision=precision)
    assert st == binding.FP9_ERR_RANGE


def test_moe_prefill_full_size_dsv3():
    """The pages' long prompt (1481 tokens) through a DeepSeek-V3 layer
    (256 routed + 1 shared expert, 12.7 GB), in both precisions: every
    token's routing against the oracle, and the outputs of sampled tokens."""
    shape = synth.DSV3
    m = 1481
    layer = support.build_layer(shape, base=41)
    ol = support.OracleLayer(shape, base=41)
    x = support.safe_tokens(shape, ol.w_router, m, base=41)
    xr = x.numpy().astype(np.float64)
    rid, rw = ol.route(xr)
    rows = [0, 1, 127, 128, 700, 1023, m - 2, m - 1]
    ref = O.moe(xr[rows], **ol.kwargs())
    for precision in (SPLIT, FP16):
        y, ids, w, st = _run(layer, x.cuda(), precision=precision)
        assert st == 0
        assert np.array_equal(ids.cpu().numpy(), rid)
        assert np.abs(w.cpu().numpy() - rw).max() <= 1e-5 * shape.route_scale
        if precision == SPLIT:
            err = support.max_rel_err(y.cpu().numpy()[rows], ref)
            assert err <= support.TOL, err
        else:
            fro, row = support.prefill_errors(y.cpu().numpy()[rows], ref)
            assert fro <= support.PREFILL_FRO and row <= support.PREFILL_ROW
        assert np.isfinite(y.cpu().numpy()).all()
