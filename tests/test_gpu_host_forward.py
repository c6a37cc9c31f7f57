"""fp9_moe_forward_host: the MoE forward with x and y in host memory (copy
in, forward, copy out, queued on one stream). It runs the same kernels on
the same inputs as fp9_moe_forward, whose parity with the oracle the other
tests check, so its y must equal the device call's bit for bit, with pinned
and with pageable host buffers, on two calls in a row."""

import pytest
import torch

from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,bsz", [(synth.TINY, 1), (synth.TINY, 3), (synth.DSV3, 1), (synth.DSV3, 2)],
                         ids=["tiny-1", "tiny-3", "dsv3-1", "dsv3-2"])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_forward_equals_device_forward(shape, bsz, pinned):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = support.build_layer(shape, base=950 + bsz, status=status)
    wr = L.w_router.cpu().numpy()
    ws = Workspace.for_moe(L, bsz)
    wsh = Workspace.for_moe_host(L, bsz)
    assert wsh.tensor.numel() >= ws.tensor.numel() + 2 * 4 * bsz * shape.hidden
    for call in range(2):
        x = support.safe_tokens(shape, wr, bsz, 960 + 10 * call + bsz, device="cuda")
        y_ref = torch.empty_like(x)
        binding.fp9_moe_forward(L, x, y_ref, ws.tensor, status)
        xh = x.cpu()
        yh = torch.full((bsz, shape.hidden), float("nan"), dtype=torch.float32)
        if pinned:
            xh, yh = xh.pin_memory(), yh.pin_memory()
        binding.fp9_moe_forward_host(L, xh, yh, wsh.tensor, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, binding.status_str(int(status.item()))
        assert torch.equal(yh, y_ref.cpu())
    del L
    torch.cuda.empty_cache()


def test_host_forward_rejects_a_short_workspace_and_device_tensors():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = support.build_layer(synth.TINY, base=990, status=status)
    xh = torch.zeros((1, synth.TINY.hidden), dtype=torch.float32).pin_memory()
    yh = torch.zeros_like(xh).pin_memory()
    short = Workspace.for_moe(L, 1)  # the forward's own workspace, without the staging rows
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_moe_forward_host(L, xh, yh, short.tensor, status)
    assert e.value.code == binding.FP9_ERR_WORKSPACE
    with pytest.raises(ValueError):
        binding.fp9_moe_forward_host(L, xh.cuda(), yh, Workspace.for_moe_host(L, 1).tensor, status)


def test_prepared_host_forward_equals_the_generic_call():
    """binding.host_forward_fn (arguments marshalled once, for per-step
    loops) runs the same call: y equal bit for bit over several steps, and
    the same error for a short workspace."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = synth.TINY
    L = support.build_layer(shape, base=995, status=status)
    wsh = Workspace.for_moe_host(L, 2)
    f = binding.host_forward_fn(L, wsh.tensor, status)
    wr = L.w_router.cpu().numpy()
    for step in range(3):
        xh = support.safe_tokens(shape, wr, 2, 996 + step).pin_memory()
        y1 = torch.empty((2, shape.hidden), dtype=torch.float32).pin_memory()
        y2 = torch.empty_like(y1).pin_memory()
        f(xh, y1)
        binding.fp9_moe_forward_host(L, xh, y2, wsh.tensor, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(y1, y2)
    g = binding.host_forward_fn(L, Workspace.for_moe(L, 2).tensor, status)
    with pytest.raises(binding.Fp9Error) as e:
        g(xh, y1)
    assert e.value.code == binding.FP9_ERR_WORKSPACE
