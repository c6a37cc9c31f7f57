"""The allocation-free MoE forward, for callers that cannot allocate device
memory (a runtime that owns and caps device memory, a plugin handed only
its buffers, a path that must not risk an allocation's synchronisation).

It runs the same kernels, plan and grid as fp9_moe_forward with the
library's fixed scratch array as the workspace, and both add their partial
sums in the same fixed order; so its routing and its output must equal the
workspace version's bit for bit, on two calls in a row (the second call
reuses the array as the first left it). Collected last, so a failure here stops a run only after
every other test has run."""

import numpy as np
import pytest
import torch

from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,bsz", [(synth.TINY, 1), (synth.TINY, 2), (synth.DSV3, 1), (synth.DSV3, 2)],
                         ids=["tiny-1", "tiny-2", "dsv3-1", "dsv3-2"])
def test_noalloc_forward_matches_workspace_forward_twice(shape, bsz):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = support.build_layer(shape, base=900 + bsz, status=status)
    wr = L.w_router.cpu().numpy()
    ws = Workspace.for_moe(L, bsz)
    for call in range(2):
        x = support.safe_tokens(shape, wr, bsz, 910 + 10 * call + bsz, device="cuda")
        y_ref = torch.empty_like(x)
        ids_ref = torch.empty((bsz, shape.topk), dtype=torch.int32, device="cuda")
        w_ref = torch.empty((bsz, shape.topk), dtype=torch.float32, device="cuda")
        binding.fp9_moe_forward(L, x, y_ref, ws.tensor, status, ids_ref, w_ref)
        y = torch.full_like(x, float("nan"))
        ids = torch.empty_like(ids_ref)
        w = torch.full_like(w_ref, float("nan"))
        binding.fp9_moe_forward_noalloc(L, x, y, status, ids, w)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, binding.status_str(int(status.item()))
        assert torch.equal(ids, ids_ref)
        assert torch.equal(w, w_ref)
        assert torch.equal(y, y_ref)
        # and the oracle's tolerance, as for the workspace call
        assert support.max_rel_err(y.cpu().numpy(), y_ref.cpu().numpy()) <= support.TOL
    del L
    torch.cuda.empty_cache()


def test_noalloc_forward_rejects_a_workspace_beyond_the_fixed_array():
    assert binding.noalloc_scratch_bytes() == 16 << 20
    shape = synth.DSV3
    L = support.build_layer(synth.DSV3, base=950)
    x = torch.zeros((8, shape.hidden), device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_moe_forward_noalloc(L, x, y)   # bsz 8 needs about 37 MB of partials
    assert e.value.code == binding.FP9_ERR_WORKSPACE
    del L
    torch.cuda.empty_cache()
