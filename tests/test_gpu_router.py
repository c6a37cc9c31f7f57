"""GPU parity for moe_router: expert ids bit-exact, weights within 1e-5 *
route_scale, on tokens whose routing margin is at least 1e-4."""

import numpy as np
import pytest
import torch

from fp9_weight_expert_gb300 import Workspace, binding, layers, synth
from tests import support

pytestmark = pytest.mark.gpu

GROUPED = synth.MoEShape(hidden=512, inter=64, n_experts=64, n_groups=8, topk_groups=3, topk=6,
                         n_shared=1, route_scale=2.5, router_std=0.05 * (64 / 512) ** 0.5)


def _router_only_layer(shape, base):
    L = layers.MoELayer(shape.hidden, shape.inter, shape.n_experts, shape.n_groups,
                        shape.topk_groups, shape.topk, shape.n_shared, shape.route_scale)
    L.w_router.copy_(support.router_source(shape, base, 0, "cuda"))
    return L


@pytest.mark.parametrize("shape", [synth.TINY, GROUPED, synth.DSV3], ids=["tiny", "grouped", "dsv3"])
@pytest.mark.parametrize("bsz", [1, 2, 5, 8])
def test_router_matches_oracle(shape, bsz):
    base = 100 + bsz
    L = _router_only_layer(shape, base)     # expert banks are not read by the router
    wr = L.w_router.cpu().numpy()
    x = support.safe_tokens(shape, wr, bsz, base, device="cuda")
    ids = torch.empty((bsz, shape.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((bsz, shape.topk), dtype=torch.float32, device="cuda")
    ws = Workspace.for_moe(L, bsz)
    binding.moe_router(L, x, ids, w, ws.tensor)
    torch.cuda.synchronize()
    import oracle as O
    rid, rw = O.route(x.cpu().numpy(), wr, shape.n_groups, shape.topk_groups, shape.topk,
                      shape.route_scale)
    assert np.array_equal(ids.cpu().numpy(), rid)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(wg - rw)) <= 1e-5 * shape.route_scale
    assert np.max(np.abs(wg.sum(axis=1) - shape.route_scale)) <= 1e-5 * shape.route_scale
    # the ticket is left at zero, so a second call works on the same workspace
    binding.moe_router(L, x, ids, w, ws.tensor)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), rid)
