"""GPU checks of fp9_moe_forward_residual, a stack's layer step with the
residual add and the RMSNorm folded into the layer's kernels: per layer,
teacher-forced against the oracle (the layer's input is the oracle's
RMSNorm of the GPU's h); end to end against the oracle's stack and the
glue path (fp9_residual_rmsnorm + fp9_moe_forward); the partial sums of
squares against float64 sums; and its CUDA-graph replay against eager."""

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _layers(shape, base, n):
    Ls = [support.build_layer(shape, base=base, layer=l) for l in range(n)]
    Os = [support.OracleLayer(shape, base=base, layer=l) for l in range(n)]
    return Ls, Os


def _check_parts(h, ss):
    """ss[t, b] is the sum of the squares of h[t, 16 b .. 16 b + 15]."""
    hh = h.cpu().numpy().astype(np.float64)
    ref = (hh * hh).reshape(hh.shape[0], -1, 16).sum(axis=2)
    assert np.abs(ss.cpu().numpy() - ref).max() <= 1e-6 * ref.max()


@pytest.mark.parametrize("bsz", [1, 2, 5, 8])
def test_residual_steps_match_oracle(bsz):
    shape = synth.TINY
    Ls, Os = _layers(shape, 80, 3)
    h = support.safe_tokens(shape, Os[0].w_router, bsz, 81, device="cuda") * 2.0
    h_in = h.cpu().numpy().astype(np.float64)
    x = torch.empty_like(h)
    ss = torch.empty((bsz, shape.hidden // 16), dtype=torch.float32, device="cuda")
    ws = Workspace.for_moe(Ls[0], bsz)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_residual_rmsnorm(h, None, x, EPS)
    checked = 0
    for l in range(3):
        hb = h.cpu().numpy().astype(np.float64)
        ids = torch.empty((bsz, shape.topk), dtype=torch.int32, device="cuda")
        binding.fp9_moe_forward_residual(Ls[l], x if l == 0 else None, h, ss, ws.tensor, status, ids, eps=EPS,
                                         next_layer=Ls[l + 1] if l + 1 < 3 else None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _check_parts(h, ss)
        # teacher-forced: the oracle's layer on the oracle's norm of this
        # layer's GPU input h (for the first layer, the glue kernel's x)
        xr = O.rmsnorm(hb, EPS)
        if np.all(Os[l].margin(xr) >= support.MARGIN_MIN):
            rid, _ = Os[l].route(xr)
            assert np.array_equal(ids.cpu().numpy(), rid)
            ref = O.moe(xr, **Os[l].kwargs())
            y = h.cpu().numpy().astype(np.float64) - hb    # h + y, rounded once to fp32
            bound = support.TOL * np.abs(ref).max(axis=1) + 2.0 ** -23 * np.abs(hb).max(axis=1)
            assert np.all(np.abs(y - ref).max(axis=1) <= bound)
            checked += 1
    assert checked >= 1
    ref_h = O.stack(h_in, [o.kwargs() for o in Os], EPS)
    assert support.max_rel_err(h.cpu().numpy(), ref_h) <= 1e-3   # end-to-end drift, as the glue path


@pytest.mark.parametrize("shape_name,bsz", [("tiny", 2), ("tiny", 5), ("dsv3", 1), ("dsv3", 2)])
def test_residual_steps_match_the_glue_path(shape_name, bsz):
    """The same layers through the glue path: the same routing, and h
    within rounding (the norm's sum of squares is added in another order)."""
    shape = synth.TINY if shape_name == "tiny" else synth.DSV3
    n = 3 if shape_name == "tiny" else 2
    Ls, Os = _layers(shape, 90, n)
    h0 = support.safe_tokens(shape, Os[0].w_router, bsz, 91, device="cuda") * 2.0
    ws = Workspace.for_moe(Ls[0], bsz)
    ids_g = torch.empty((n, bsz, shape.topk), dtype=torch.int32, device="cuda")
    ids_r = torch.empty_like(ids_g)
    hg = h0.clone()
    x = torch.empty_like(hg)
    y = torch.empty_like(hg)
    binding.fp9_residual_rmsnorm(hg, None, x, EPS)
    margins = []
    for l, L in enumerate(Ls):
        margins.append(Os[l].margin(x.cpu().numpy()))
        binding.fp9_moe_forward(L, x, y, ws.tensor, None, ids_g[l])
        binding.fp9_residual_rmsnorm(hg, y, x, EPS)
    hr = h0.clone()
    ss = torch.empty((bsz, shape.hidden // 16), dtype=torch.float32, device="cuda")
    binding.fp9_residual_rmsnorm(hr, None, x, EPS)
    for l, L in enumerate(Ls):
        binding.fp9_moe_forward_residual(L, x if l == 0 else None, hr, ss, ws.tensor, None, ids_r[l], eps=EPS)
    torch.cuda.synchronize()
    if all(np.all(m >= support.MARGIN_MIN) for m in margins):
        assert torch.equal(ids_r, ids_g)
        assert support.max_rel_err(hr.cpu().numpy(), hg.cpu().numpy()) <= 1e-5
    else:   # a near-tie may route differently: only the first layer is compared
        assert torch.equal(ids_r[0], ids_g[0])
    _check_parts(hr, ss)


def test_residual_stack_in_a_cuda_graph_matches_eager():
    shape, bsz = synth.TINY, 2
    Ls, Os = _layers(shape, 95, 3)
    h0 = support.safe_tokens(shape, Os[0].w_router, bsz, 96, device="cuda") * 2.0
    ws = Workspace.for_moe(Ls[0], bsz)
    h = h0.clone()
    x = torch.empty_like(h)
    ss = torch.empty((bsz, shape.hidden // 16), dtype=torch.float32, device="cuda")

    def run():
        binding.fp9_residual_rmsnorm(h, None, x, EPS)
        for l, L in enumerate(Ls):
            binding.fp9_moe_forward_residual(L, x if l == 0 else None, h, ss, ws.tensor, eps=EPS,
                                             next_layer=Ls[(l + 1) % 3])

    run()
    torch.cuda.synchronize()
    eager, eager_ss = h.clone(), ss.clone()
    run()   # again from the updated h: a second eager pass is deterministic too
    torch.cuda.synchronize()
    second = h.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        h.copy_(h0)
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        h.copy_(h0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(h, eager) and torch.equal(ss, eager_ss)
    h.copy_(eager)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(h, second)
