"""ctypes binding of libfp9moe.so: one Python function per C entry point,
same names, argument marshalling only. Every step of the path runs in the
library's CUDA kernels; there is no fallback. If the library is missing,
loading raises.

Tensors are torch tensors on the current CUDA device; the work is queued on
torch's current stream unless ``stream`` (a torch.cuda.Stream) is given.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build_lib

FP9_OK = 0
FP9_ERR_INVALID_ARG = 1
FP9_ERR_SHAPE = 2
FP9_ERR_ALIGN = 3
FP9_ERR_WORKSPACE = 4
FP9_ERR_RANGE = 5
FP9_ERR_CUDA = 6
FP9_ERR_TIMEOUT = 7

FP9_PREFILL_SPLIT = 0   # prefill activations as two fp16 terms (hi + lo): the default
FP9_PREFILL_FP16 = 1    # one fp16 term per activation: faster, looser

FP9_MAX_BSZ = 8
FP9_MAX_HIDDEN = 7168
FP9_MAX_PREFILL_TOKENS = 1048576
FP9_MAX_PREFILL_HIDDEN = 32768


class Fp9Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_str(code)}")


class FFNBankC(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_int64),
        ("inter", ctypes.c_int64),
        ("hidden", ctypes.c_int64),
        ("gate_body", ctypes.c_void_p),
        ("gate_sign", ctypes.c_void_p),
        ("up_body", ctypes.c_void_p),
        ("up_sign", ctypes.c_void_p),
        ("down_body", ctypes.c_void_p),
        ("down_sign", ctypes.c_void_p),
    ]


class MoELayerC(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int64),
        ("inter", ctypes.c_int64),
        ("n_experts", ctypes.c_int32),
        ("n_groups", ctypes.c_int32),
        ("topk_groups", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("n_shared", ctypes.c_int32),
        ("route_scale", ctypes.c_float),
        ("w_router", ctypes.c_void_p),
        ("routed", FFNBankC),
        ("shared", FFNBankC),
    ]


_LIB = None

_SIGS = {
    "fp9_pack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_from_fp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_moe_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(MoELayerC), ctypes.c_int32]),
    "fp9_dense_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(FFNBankC), ctypes.c_int32]),
    "moe_router": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_int32,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p]),
    "fp9_moe_forward": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                       ctypes.c_void_p]),
    "fp9_moe_forward_residual": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_int32, ctypes.c_float,
                                                ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_dense_ffn": (ctypes.c_int, [ctypes.POINTER(FFNBankC), ctypes.c_void_p, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_residual_rmsnorm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                            ctypes.c_void_p]),
    "fp9_selftest_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                            ctypes.c_int32, ctypes.c_void_p]),
    "fp9_status_str": (ctypes.c_char_p, [ctypes.c_int32]),
    "fp9_profile_events": (None, [ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_moe_forward_host": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                            ctypes.c_void_p]),
    "fp9_moe_host_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(MoELayerC), ctypes.c_int32]),
    "fp9_moe_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_moe_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "fp9_ffn_prefill": (ctypes.c_int, [ctypes.POINTER(FFNBankC), ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(FFNBankC), ctypes.c_int64]),
    "fp9_moe_prefill": (ctypes.c_int, [ctypes.POINTER(MoELayerC), ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "fp9_moe_prefill_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(MoELayerC), ctypes.c_int64]),
    "fp9_prefill_selftest_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                    ctypes.c_int32, ctypes.c_void_p]),
}


def lib_path() -> str:
    return build_lib.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libfp9moe.so (built by ``build_lib.build()``); raises if absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libfp9moe.so not found at {p}: build it with "
                           "`python -m fp9_weight_expert_gb300.build_lib` (needs nvcc)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def status_str(code: int) -> str:
    return load().fp9_status_str(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != FP9_OK:
        raise Fp9Error(code, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------- entry points

def fp9_pack(src: torch.Tensor, body: torch.Tensor, sign: torch.Tensor,
             status: torch.Tensor | None = None, stream=None) -> None:
    """Encodes fp32 [rows, cols] into body [rows, cols] and sign [rows, cols/8]."""
    rows, cols = src.shape[-2], src.shape[-1]
    rows = src.numel() // cols if cols else 0
    _check(load().fp9_pack(_ptr(src), rows, cols, _ptr(body), _ptr(sign), _ptr(status),
                           _stream(stream)), "fp9_pack")


def fp9_from_fp8(w8: torch.Tensor, scale_inv: torch.Tensor, body: torch.Tensor, sign: torch.Tensor,
                 status: torch.Tensor | None = None, stream=None) -> None:
    """Converts fp8 e4m3 bytes [rows, cols] (uint8) with fp32 block scales
    [ceil(rows/128), ceil(cols/128)] into body [rows, cols] and sign [rows, cols/8]."""
    rows, cols = w8.shape[-2], w8.shape[-1]
    _check(load().fp9_from_fp8(_ptr(w8), _ptr(scale_inv), rows, cols, _ptr(body), _ptr(sign), _ptr(status),
                               _stream(stream)), "fp9_from_fp8")


def fp9_decode(body: torch.Tensor, sign: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    cols = body.shape[-1]
    rows = body.numel() // cols if cols else 0
    _check(load().fp9_decode(_ptr(body), _ptr(sign), rows, cols, _ptr(dst), _stream(stream)),
           "fp9_decode")


def moe_workspace_bytes(layer, bsz: int) -> int:
    return int(load().fp9_moe_workspace_bytes(ctypes.byref(layer.c_struct()), bsz))


def moe_host_workspace_bytes(layer, bsz: int) -> int:
    return int(load().fp9_moe_host_workspace_bytes(ctypes.byref(layer.c_struct()), bsz))


def dense_workspace_bytes(ffn, bsz: int) -> int:
    return int(load().fp9_dense_workspace_bytes(ctypes.byref(ffn.c_struct()), bsz))


def moe_router(layer, x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor,
               ws: torch.Tensor, stream=None) -> None:
    _check(load().moe_router(ctypes.byref(layer.c_struct()), _ptr(x), x.shape[0], _ptr(ids),
                             _ptr(weights), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "moe_router")


def fp9_moe_forward(layer, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                    status: torch.Tensor | None = None, ids: torch.Tensor | None = None,
                    weights: torch.Tensor | None = None, stream=None) -> None:
    _check(load().fp9_moe_forward(ctypes.byref(layer.c_struct()), _ptr(x), x.shape[0], _ptr(y),
                                  _ptr(ids), _ptr(weights), _ptr(ws),
                                  ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "fp9_moe_forward")


def fp9_moe_forward_residual(layer, x: torch.Tensor | None, h: torch.Tensor, ss: torch.Tensor, ws: torch.Tensor,
                             status: torch.Tensor | None = None, ids: torch.Tensor | None = None,
                             weights: torch.Tensor | None = None, eps: float = 1e-6, next_layer=None,
                             stream=None) -> None:
    """One layer step of a stack: h += MoE(x), or h += MoE(RMSNorm(h))
    when x is None (the norm's sums of squares come from ss, which the call
    then rewrites for the new h: [bsz, hidden / 16] fp32). next_layer: the
    stack's next layer, whose router weights are read into L2."""
    nxt = ctypes.byref(next_layer.c_struct()) if next_layer is not None else None
    _check(load().fp9_moe_forward_residual(ctypes.byref(layer.c_struct()), _ptr(x), _ptr(h), _ptr(ss), h.shape[0],
                                           ctypes.c_float(eps), nxt, _ptr(ids), _ptr(weights), _ptr(ws),
                                           ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "fp9_moe_forward_residual")


def fp9_moe_forward_host(layer, x_host: torch.Tensor, y_host: torch.Tensor, ws: torch.Tensor,
                         status: torch.Tensor | None = None, stream=None) -> None:
    """fp9_moe_forward with x and y in host memory (pinned CPU tensors for
    asynchronous copies): queues the copy in, the forward and the copy out;
    y_host holds the result once the stream is synchronised."""
    if x_host.device.type != "cpu" or y_host.device.type != "cpu":
        raise ValueError("fp9_moe_forward_host takes host (CPU) tensors for x and y")
    _check(load().fp9_moe_forward_host(ctypes.byref(layer.c_struct()), _ptr(x_host), x_host.shape[0],
                                       _ptr(y_host), _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                       _stream(stream)), "fp9_moe_forward_host")


def host_forward_fn(layer, ws: torch.Tensor, status: torch.Tensor | None = None, stream=None):
    """fp9_moe_forward_host with the layer, the workspace, the status word and
    the stream marshalled once: returns f(x_host, y_host) for a per-step
    loop, which passes only the two host buffers' addresses per call (the
    generic wrapper spends some microseconds of Python per call on
    argument conversion). x_host, y_host: pinned CPU tensors [bsz, hidden]."""
    fn = load().fp9_moe_forward_host
    lp = ctypes.byref(layer.c_struct())
    wp, wn, sp, st = _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream)

    def call(x_host: torch.Tensor, y_host: torch.Tensor) -> None:
        code = fn(lp, x_host.data_ptr(), x_host.shape[0], y_host.data_ptr(), wp, wn, sp, st)
        if code != FP9_OK:
            raise Fp9Error(code, "fp9_moe_forward_host")
    return call


def fp9_dense_ffn(ffn, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                  status: torch.Tensor | None = None, stream=None) -> None:
    _check(load().fp9_dense_ffn(ctypes.byref(ffn.c_struct()), _ptr(x), x.shape[0], _ptr(y),
                                _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                _stream(stream)), "fp9_dense_ffn")


def fp9_residual_rmsnorm(h: torch.Tensor, y: torch.Tensor | None, x_out: torch.Tensor,
                         eps: float = 1e-6, stream=None) -> None:
    _check(load().fp9_residual_rmsnorm(_ptr(h), _ptr(y), _ptr(x_out), h.shape[0], h.shape[1],
                                       eps, _stream(stream)), "fp9_residual_rmsnorm")


def fp9_selftest_timeout(ws: torch.Tensor, status: torch.Tensor, timeout_us: int = 2000,
                         stream=None) -> None:
    _check(load().fp9_selftest_timeout(_ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                       timeout_us, _stream(stream)), "fp9_selftest_timeout")


def fp9_profile_events(start, stop) -> None:
    """Brackets every later fused-kernel launch with two torch.cuda.Events
    (recorded on the kernel's stream); (None, None) turns it off. Each event
    must have been recorded once, so that torch has created it."""
    if start is not None and (start.cuda_event == 0 or stop.cuda_event == 0):
        raise ValueError("record each event once before passing it (torch creates it lazily)")
    load().fp9_profile_events(start.cuda_event if start is not None else None,
                              stop.cuda_event if stop is not None else None)


def fp9_moe_forward_noalloc(layer, x: torch.Tensor, y: torch.Tensor, status: torch.Tensor | None = None,
                            ids: torch.Tensor | None = None, weights: torch.Tensor | None = None,
                            stream=None) -> None:
    """fp9_moe_forward without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed scratch array is used
    instead (see include/fp9moe.h for its size and sharing rules)."""
    _check(load().fp9_moe_forward_noalloc(ctypes.byref(layer.c_struct()), _ptr(x), x.shape[0], _ptr(y),
                                          _ptr(ids), _ptr(weights), _ptr(status), _stream(stream)),
           "fp9_moe_forward_noalloc")


def noalloc_scratch_bytes() -> int:
    return int(load().fp9_moe_noalloc_scratch_bytes())


def prefill_workspace_bytes(ffn, m: int) -> int:
    return int(load().fp9_prefill_workspace_bytes(ctypes.byref(ffn.c_struct()), m))


def fp9_ffn_prefill(ffn, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor, k: int = 0,
                    status: torch.Tensor | None = None, stream=None, precision: int = FP9_PREFILL_SPLIT) -> None:
    """y [m, hidden] = FFN k of the bank ``ffn`` applied to x [m, hidden]
    (fp32), on the tensor cores (x and h as two fp16 terms each by default,
    or one with FP9_PREFILL_FP16; fp32 accumulation)."""
    _check(load().fp9_ffn_prefill(ctypes.byref(ffn.c_struct()), k, _ptr(x), x.shape[0], _ptr(y), precision,
                                  _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream)),
           "fp9_ffn_prefill")


def moe_prefill_workspace_bytes(layer, m: int) -> int:
    return int(load().fp9_moe_prefill_workspace_bytes(ctypes.byref(layer.c_struct()), m))


def fp9_moe_prefill(layer, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor,
                    status: torch.Tensor | None = None, ids: torch.Tensor | None = None,
                    weights: torch.Tensor | None = None, stream=None, precision: int = FP9_PREFILL_SPLIT) -> None:
    """y [m, hidden] = the MoE layer applied to m tokens x (fp32) at once,
    expert FFNs on the tensor cores (activations as two fp16 terms by
    default, or one with FP9_PREFILL_FP16; fp32 accumulation)."""
    _check(load().fp9_moe_prefill(ctypes.byref(layer.c_struct()), _ptr(x), x.shape[0], _ptr(y), _ptr(ids),
                                  _ptr(weights), precision, _ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                  _stream(stream)), "fp9_moe_prefill")


def fp9_prefill_selftest_timeout(ws: torch.Tensor, status: torch.Tensor, timeout_us: int = 2000,
                                 stream=None) -> None:
    _check(load().fp9_prefill_selftest_timeout(_ptr(ws), ws.numel() * ws.element_size(), _ptr(status),
                                               timeout_us, _stream(stream)), "fp9_prefill_selftest_timeout")
