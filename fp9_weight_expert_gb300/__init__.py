"""fp9 FFN/MoE decode step (and FFN prefill) for GB300 (sm_103a).

The compute path is libfp9moe.so (hand-written CUDA kernels behind a C ABI,
declared in include/fp9moe.h); this package holds its build step, a ctypes
binding with the same entry-point names, containers for fp9 weights resident
in HBM, and seeded synthetic input generators.
"""

from . import binding, build_lib, layers, synth  # noqa: F401
from .binding import (  # noqa: F401
    Fp9Error, fp9_decode, fp9_dense_ffn, fp9_ffn_prefill, fp9_from_fp8, fp9_moe_forward, fp9_moe_forward_residual, fp9_moe_prefill, fp9_pack,
    fp9_residual_rmsnorm, fp9_selftest_timeout, moe_router, status_str,
)
from .layers import FFNBank, MoELayer, Workspace  # noqa: F401

__all__ = [
    "binding", "build_lib", "layers", "synth", "Fp9Error", "fp9_pack", "fp9_decode", "moe_router",
    "fp9_moe_forward", "fp9_moe_forward_residual", "fp9_dense_ffn", "fp9_ffn_prefill", "fp9_moe_prefill", "fp9_from_fp8", "fp9_residual_rmsnorm", "fp9_selftest_timeout",
    "status_str", "FFNBank", "MoELayer", "Workspace",
]
