"""GPU parity for fp9_moe_forward against the oracle: routing ids bit-exact,
outputs within max|gpu - oracle| <= 2e-4 * max|oracle| per token vector.
Small layers span several chunks and a ragged tail of the intermediate
dimension; the DeepSeek-V3 layer runs at full size, in the launch
configuration the benchmark times."""

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu

# 203 = 50 full 4-row chunks + a 3-row tail; 16 experts in 4 groups, 2 shared
MID = synth.MoEShape(hidden=1024, inter=203, n_experts=16, n_groups=4, topk_groups=2, topk=4,
                     n_shared=2, route_scale=2.5, router_std=0.05 * (16 / 1024) ** 0.5)
# 128-wide hidden (the smallest allowed), 1-row intermediate: every chunk is a tail
NARROW = synth.MoEShape(hidden=128, inter=1, n_experts=8, n_groups=2, topk_groups=1, topk=3,
                        n_shared=0, route_scale=1.0, router_std=0.05)
# fewer (job, row) pairs than SMs: each job spans several one-row CTAs
FEWROWS = synth.MoEShape(hidden=256, inter=5, n_experts=8, n_groups=1, topk_groups=1, topk=3,
                         n_shared=1, route_scale=1.0, router_std=0.05)
# about as many rows as SMs: CTAs own one or two rows across job boundaries
NEARSM = synth.MoEShape(hidden=384, inter=37, n_experts=16, n_groups=2, topk_groups=1, topk=3,
                        n_shared=1, route_scale=1.0, router_std=0.05 * (16 / 384) ** 0.5)
# more than 256 experts (32 per lane in the one-warp routing), 16 groups of 40, top-6
WIDE = synth.MoEShape(hidden=256, inter=24, n_experts=640, n_groups=16, topk_groups=5, topk=6,
                      n_shared=1, route_scale=2.0, router_std=0.05)


def _run(shape, bsz, base, layer=None, ol=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = layer or support.build_layer(shape, base=base, status=status)
    ol = ol or support.OracleLayer(shape, base=base)
    x = support.safe_tokens(shape, ol.w_router, bsz, base + 17, device="cuda")
    y = torch.full_like(x, float("nan"))
    ids = torch.empty((bsz, shape.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((bsz, shape.topk), dtype=torch.float32, device="cuda")
    ws = Workspace.for_moe(L, bsz)
    binding.fp9_moe_forward(L, x, y, ws.tensor, status, ids, w)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, binding.status_str(int(status.item()))
    return L, ol, x, y, ids, w, ws, status


@pytest.mark.parametrize("shape", [synth.TINY, MID, NARROW, FEWROWS, NEARSM, WIDE],
                         ids=["tiny", "mid", "narrow", "fewrows", "nearsm", "wide"])
@pytest.mark.parametrize("bsz", [1, 2, 3, 5, 8])
def test_moe_forward_matches_oracle(shape, bsz):
    L, ol, x, y, ids, w, ws, status = _run(shape, bsz, base=200 + bsz)
    xr = x.cpu().numpy()
    rid, rw = ol.route(xr)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.max(np.abs(w.cpu().numpy() - rw)) <= 1e-5 * shape.route_scale
    ref = O.moe(xr, **ol.kwargs())
    err = support.max_rel_err(y.cpu().numpy(), ref)
    assert err <= support.TOL, err
    # same workspace again: deterministic, bit-identical output
    y2 = torch.empty_like(y)
    binding.fp9_moe_forward(L, x, y2, ws.tensor, status)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_moe_forward_zero_routed_experts_gives_shared_only():
    shape = MID
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = support.build_layer(shape, base=300, status=status)
    for m in range(3):
        L.routed.body[m].zero_()
        L.routed.sign[m].zero_()
    ol = support.OracleLayer(shape, base=300)
    x = support.safe_tokens(shape, ol.w_router, 3, 301, device="cuda")
    y = torch.empty_like(x)
    binding.fp9_moe_forward(L, x, y, Workspace.for_moe(L, 3).tensor, status)
    torch.cuda.synchronize()
    ref = sum(O.dense_ffn(x.cpu().numpy(), ol.planes(1, k)) for k in range(shape.n_shared))
    assert support.max_rel_err(y.cpu().numpy(), ref) <= support.TOL


def test_moe_forward_rejects_bad_arguments():
    shape = synth.TINY
    L = support.build_layer(shape, base=5)
    x = torch.zeros((2, shape.hidden), device="cuda")
    y = torch.empty_like(x)
    ws = Workspace.for_moe(L, 2)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_moe_forward(L, x, y, small)
    assert e.value.code == binding.FP9_ERR_WORKSPACE
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_moe_forward(L, torch.zeros((9, shape.hidden), device="cuda"),
                                torch.zeros((9, shape.hidden), device="cuda"), ws.tensor)
    assert e.value.code == binding.FP9_ERR_INVALID_ARG
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_moe_forward(L, x[:, 1:], y, ws.tensor)   # misaligned x
    assert e.value.code == binding.FP9_ERR_ALIGN


@pytest.fixture(scope="module")
def dsv3_layer():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = support.build_layer(synth.DSV3, base=11, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yield L, support.OracleLayer(synth.DSV3, base=11)
    del L
    torch.cuda.empty_cache()


@pytest.mark.parametrize("bsz", [1, 2, 5, 8])
def test_moe_forward_full_dsv3_layer(dsv3_layer, bsz):
    L, ol = dsv3_layer
    _, _, x, y, ids, w, ws, status = _run(synth.DSV3, bsz, base=400 + bsz, layer=L, ol=ol)
    xr = x.cpu().numpy()
    rid, rw = ol.route(xr)
    assert np.array_equal(ids.cpu().numpy(), rid)
    # every token of the call against the oracle
    ref = O.moe(xr, **ol.kwargs())
    err = support.max_rel_err(y.cpu().numpy(), ref)
    assert err <= support.TOL, err
