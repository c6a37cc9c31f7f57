"""Failure detection without faulting the GPU: a fused-kernel launch whose
copies are switched off runs every bounded wait out; the kernel records
FP9_ERR_TIMEOUT and returns, and the context stays usable."""

import pytest
import torch

from fp9_weight_expert_gb300 import Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_selftest_timeout(ws, status, timeout_us=2000)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.FP9_ERR_TIMEOUT
    # the context still works: a real forward afterwards is correct
    shape = synth.TINY
    L = support.build_layer(shape, base=3)
    ol = support.OracleLayer(shape, base=3)
    x = support.safe_tokens(shape, ol.w_router, 1, 4, device="cuda")
    y = torch.empty_like(x)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_moe_forward(L, x, y, Workspace.for_moe(L, 1).tensor, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    import oracle as O
    ref = O.moe(x.cpu().numpy(), **ol.kwargs())
    assert support.max_rel_err(y.cpu().numpy(), ref) <= support.TOL


def test_selftest_rejects_bad_arguments():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_selftest_timeout(small, status)
    assert e.value.code == binding.FP9_ERR_WORKSPACE


def test_prefill_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(1 << 17, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_prefill_selftest_timeout(ws, status, timeout_us=2000)
    torch.cuda.synchronize()
    assert int(status.item()) == binding.FP9_ERR_TIMEOUT
    # the context still works: a real prefill afterwards is correct
    import numpy as np

    import oracle as O
    from fp9_weight_expert_gb300 import FFNBank
    f = FFNBank(1, 128, 256)
    dec = []
    for m in range(3):
        w = synth.ffn_weight(None, 128, 256, synth.seed_for(12, 0, synth.DENSE, 0, m), "cuda")
        f.pack(0, m, w)
        b, s_, _ = O.fp9_pack(w.cpu().numpy())
        dec.append(O.fp9_decode(b, s_))
    x = synth.tokens(100, 256, 13, "cuda")
    y = torch.empty_like(x)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_ffn_prefill(f, x, y, Workspace.for_prefill(f, 100).tensor, 0, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    support.check_prefill(y.cpu().numpy(), x.cpu().numpy().astype(np.float64), *dec)
