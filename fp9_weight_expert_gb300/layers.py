"""Containers that hold fp9 weights resident in HBM and describe them to the
C ABI. They allocate torch tensors (the library itself allocates nothing)
and fill them with the library's fp9_pack kernel; all compute goes through
``binding``.

Layout in HBM (one allocation per plane of a bank):
  gate/up/down body  uint8 [n, inter, hidden]
  gate/up/down sign  uint8 [n, inter, hidden / 8]
down is stored transposed (down_t = W_down^T) so that the down weights of
one intermediate row are contiguous; a DeepSeek-V3 MoE layer (256 routed +
1 shared expert of 3 x 2048 x 7168) takes 12.73 GB.
"""

from __future__ import annotations

import ctypes
from typing import Callable

import torch

from . import binding

GATE, UP, DOWN_T = 0, 1, 2
_PLANES = ("gate", "up", "down")


class FFNBank:
    """n SwiGLU FFNs of shape [inter, hidden] in fp9 planes."""

    def __init__(self, n: int, inter: int, hidden: int, device="cuda"):
        if hidden % 8:
            raise ValueError("hidden must be a multiple of 8")
        self.n, self.inter, self.hidden = int(n), int(inter), int(hidden)
        self.body = [torch.empty((n, inter, hidden), dtype=torch.uint8, device=device) for _ in range(3)]
        self.sign = [torch.empty((n, inter, hidden // 8), dtype=torch.uint8, device=device) for _ in range(3)]
        self._c = None

    def c_struct(self) -> binding.FFNBankC:
        if self._c is None:
            self._c = binding.FFNBankC(
                self.n, self.inter, self.hidden,
                self.body[0].data_ptr(), self.sign[0].data_ptr(),
                self.body[1].data_ptr(), self.sign[1].data_ptr(),
                self.body[2].data_ptr(), self.sign[2].data_ptr())
        return self._c

    def pack(self, k: int, matrix: int, w: torch.Tensor, status=None) -> None:
        """fp9-encodes fp32 [inter, hidden] into FFN k's matrix (GATE/UP/DOWN_T)."""
        binding.fp9_pack(w, self.body[matrix][k], self.sign[matrix][k], status)

    def planes(self, k: int):
        """(gate_body, gate_sign, up_body, up_sign, down_body, down_sign) of FFN k."""
        out = []
        for m in range(3):
            out += [self.body[m][k], self.sign[m][k]]
        return tuple(out)

    def nbytes(self) -> int:
        return sum(t.numel() for t in self.body + self.sign)


class MoELayer:
    """Router weight plus routed and shared fp9 expert banks."""

    def __init__(self, hidden, inter, n_experts, n_groups, topk_groups, topk, n_shared,
                 route_scale, device="cuda"):
        self.hidden, self.inter = int(hidden), int(inter)
        self.n_experts, self.n_groups = int(n_experts), int(n_groups)
        self.topk_groups, self.topk = int(topk_groups), int(topk)
        self.n_shared, self.route_scale = int(n_shared), float(route_scale)
        self.w_router = torch.empty((n_experts, hidden), dtype=torch.float32, device=device)
        self.routed = FFNBank(n_experts, inter, hidden, device)
        self.shared = FFNBank(max(n_shared, 0), inter, hidden, device)
        self._c = None

    def c_struct(self) -> binding.MoELayerC:
        if self._c is None:
            self._c = binding.MoELayerC(
                self.hidden, self.inter, self.n_experts, self.n_groups, self.topk_groups,
                self.topk, self.n_shared, self.route_scale, self.w_router.data_ptr(),
                self.routed.c_struct(), self.shared.c_struct())
        return self._c

    def fill(self, weight: Callable[[int, int, int], torch.Tensor],
             router: torch.Tensor, status=None) -> None:
        """Packs every matrix: weight(bank, k, matrix) -> fp32 [inter, hidden]
        (bank 0 = routed, 1 = shared)."""
        self.w_router.copy_(router)
        for bank_id, bank in ((0, self.routed), (1, self.shared)):
            for k in range(bank.n):
                for m in range(3):
                    bank.pack(k, m, weight(bank_id, k, m), status)

    def nbytes(self) -> int:
        return self.routed.nbytes() + self.shared.nbytes() + self.w_router.numel() * 4


class Workspace:
    """A zeroed device workspace of at least ``nbytes`` (256-byte aligned by
    the CUDA allocator)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.tensor = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)

    @classmethod
    def for_moe(cls, layer: MoELayer, bsz: int, device="cuda"):
        n = binding.moe_workspace_bytes(layer, bsz)
        if n == 0:
            raise binding.Fp9Error(binding.FP9_ERR_INVALID_ARG, "moe_workspace_bytes")
        return cls(n, device)

    @classmethod
    def for_moe_host(cls, layer: MoELayer, bsz: int, device="cuda"):
        n = binding.moe_host_workspace_bytes(layer, bsz)
        if n == 0:
            raise binding.Fp9Error(binding.FP9_ERR_INVALID_ARG, "moe_host_workspace_bytes")
        return cls(n, device)

    @classmethod
    def for_dense(cls, ffn: FFNBank, bsz: int, device="cuda"):
        n = binding.dense_workspace_bytes(ffn, bsz)
        if n == 0:
            raise binding.Fp9Error(binding.FP9_ERR_INVALID_ARG, "dense_workspace_bytes")
        return cls(n, device)

    @classmethod
    def for_prefill(cls, ffn: FFNBank, m: int, device="cuda"):
        n = binding.prefill_workspace_bytes(ffn, m)
        if n == 0:
            raise binding.Fp9Error(binding.FP9_ERR_INVALID_ARG, "prefill_workspace_bytes")
        return cls(n, device)

    @classmethod
    def for_moe_prefill(cls, layer: MoELayer, m: int, device="cuda"):
        n = binding.moe_prefill_workspace_bytes(layer, m)
        if n == 0:
            raise binding.Fp9Error(binding.FP9_ERR_INVALID_ARG, "moe_prefill_workspace_bytes")
        return cls(n, device)
