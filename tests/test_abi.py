"""C ABI checks that need no GPU: the library builds and loads, exports
every function include/fp9moe.h declares, and its host-side argument checks
return the documented status codes before touching CUDA."""

import ctypes
import os
import re

import pytest

from fp9_weight_expert_gb300 import binding, build_lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fp9moe.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return binding.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["fp9_pack", "fp9_decode", "moe_router", "fp9_moe_forward", "fp9_dense_ffn",
              "fp9_moe_workspace_bytes", "fp9_dense_workspace_bytes", "fp9_residual_rmsnorm",
              "fp9_selftest_timeout", "fp9_status_str", "fp9_from_fp8", "fp9_ffn_prefill",
              "fp9_prefill_workspace_bytes", "fp9_moe_prefill", "fp9_moe_prefill_workspace_bytes",
              "fp9_prefill_selftest_timeout", "fp9_moe_forward_host", "fp9_moe_host_workspace_bytes",
              "fp9_moe_forward_residual"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), f"libfp9moe.so does not export {n}"


def test_status_strings(lib):
    for code in range(8):
        assert binding.status_str(code).startswith("FP9_")
    assert "unknown" in binding.status_str(99)


P = 0x100000  # a fake, 256-byte aligned "device" address: never dereferenced


def _bank(n, inter, hidden, base=P):
    return binding.FFNBankC(n, inter, hidden, base, base, base, base, base, base)


def _layer(**kw):
    d = dict(hidden=256, inter=128, n_experts=8, n_groups=1, topk_groups=1, topk=2, n_shared=1,
             route_scale=1.0)
    d.update(kw)
    return binding.MoELayerC(d["hidden"], d["inter"], d["n_experts"], d["n_groups"],
                             d["topk_groups"], d["topk"], d["n_shared"], d["route_scale"],
                             kw.get("w_router", P), kw.get("routed", _bank(d["n_experts"], d["inter"], d["hidden"])),
                             kw.get("shared", _bank(d["n_shared"], d["inter"], d["hidden"])))


def test_pack_decode_argument_checks(lib):
    assert lib.fp9_pack(P, 4, 12, P, P, None, None) == binding.FP9_ERR_SHAPE
    assert lib.fp9_pack(P, -1, 8, P, P, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_pack(None, 4, 8, P, P, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_pack(P + 4, 4, 8, P, P, None, None) == binding.FP9_ERR_ALIGN
    assert lib.fp9_pack(None, 0, 8, None, None, None, None) == binding.FP9_OK   # empty: no-op
    assert lib.fp9_decode(P, P, 4, 12, P, None) == binding.FP9_ERR_SHAPE
    assert lib.fp9_decode(P, P, 4, 8, P + 8, None) == binding.FP9_ERR_ALIGN


def test_from_fp8_argument_checks(lib):
    # (w8, scale, rows, cols, body, sign, status, stream): every case is
    # refused on the host before a device query or launch
    assert lib.fp9_from_fp8(P, P, 128, 12, P, P, None, None) == binding.FP9_ERR_SHAPE       # cols % 8
    assert lib.fp9_from_fp8(P, P, -1, 8, P, P, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_from_fp8(None, P, 128, 128, P, P, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_from_fp8(P, None, 128, 128, P, P, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_from_fp8(P, P, 128, 128, P, None, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_from_fp8(P + 4, P, 128, 128, P, P, None, None) == binding.FP9_ERR_ALIGN   # w8: 8 bytes
    assert lib.fp9_from_fp8(P, P + 2, 128, 128, P, P, None, None) == binding.FP9_ERR_ALIGN   # scales: 4
    assert lib.fp9_from_fp8(P, P, 128, 128, P + 4, P, None, None) == binding.FP9_ERR_ALIGN   # body: 8
    assert lib.fp9_from_fp8(None, None, 0, 128, None, None, None, None) == binding.FP9_OK     # empty: no-op


def _fwd(lib, layer, bsz=1, x=P, y=P + 0x10000, ws=P + 0x20000, ws_bytes=1 << 30):
    return lib.fp9_moe_forward(ctypes.byref(layer), x, bsz, y, None, None, ws, ws_bytes, None, None)


def test_moe_forward_argument_checks(lib):
    assert lib.fp9_moe_forward(None, P, 1, P, None, None, P, 1, None, None) == binding.FP9_ERR_INVALID_ARG
    assert _fwd(lib, _layer(), bsz=0) == binding.FP9_ERR_INVALID_ARG
    assert _fwd(lib, _layer(), bsz=9) == binding.FP9_ERR_INVALID_ARG
    assert _fwd(lib, _layer(hidden=200, routed=_bank(8, 128, 200), shared=_bank(1, 128, 200))) \
        == binding.FP9_ERR_SHAPE
    assert _fwd(lib, _layer(hidden=7296, routed=_bank(8, 128, 7296), shared=_bank(1, 128, 7296))) \
        == binding.FP9_ERR_SHAPE
    assert _fwd(lib, _layer(n_groups=3)) == binding.FP9_ERR_SHAPE        # 8 % 3 != 0
    assert _fwd(lib, _layer(topk=17)) == binding.FP9_ERR_SHAPE
    assert _fwd(lib, _layer(n_groups=4, topk_groups=1, topk=3)) == binding.FP9_ERR_SHAPE
    assert _fwd(lib, _layer(routed=_bank(7, 128, 256))) == binding.FP9_ERR_SHAPE
    assert _fwd(lib, _layer(routed=_bank(8, 128, 256, base=P + 8))) == binding.FP9_ERR_ALIGN
    assert _fwd(lib, _layer(w_router=P + 4)) == binding.FP9_ERR_ALIGN
    assert _fwd(lib, _layer(), x=P + 4) == binding.FP9_ERR_ALIGN
    assert _fwd(lib, _layer(), y=P) == binding.FP9_ERR_INVALID_ARG       # y aliases x
    assert _fwd(lib, _layer(), ws=P + 16) == binding.FP9_ERR_ALIGN
    assert lib.fp9_moe_workspace_bytes(ctypes.byref(_layer(topk=17)), 1) == 0


def test_moe_forward_residual_argument_checks(lib):
    L = _layer()
    H, SS, WS = P, P + 0x10000, P + 0x20000

    def call(layer=L, x=None, h=H, ss=SS, bsz=1, eps=1e-6, ws=WS, nxt=None):
        return lib.fp9_moe_forward_residual(ctypes.byref(layer) if layer is not None else None, x, h, ss, bsz,
                                            ctypes.c_float(eps), ctypes.byref(nxt) if nxt is not None else None,
                                            None, None, ws, 1 << 30, None, None)
    assert call(layer=None) == binding.FP9_ERR_INVALID_ARG
    assert call(bsz=0) == binding.FP9_ERR_INVALID_ARG
    assert call(bsz=9) == binding.FP9_ERR_INVALID_ARG
    assert call(h=None) == binding.FP9_ERR_INVALID_ARG
    assert call(ss=None) == binding.FP9_ERR_INVALID_ARG
    assert call(ws=None) == binding.FP9_ERR_INVALID_ARG
    assert call(x=H) == binding.FP9_ERR_INVALID_ARG           # x aliases h
    assert call(eps=-1.0) == binding.FP9_ERR_INVALID_ARG
    assert call(eps=2.0) == binding.FP9_ERR_INVALID_ARG
    assert call(h=H + 4) == binding.FP9_ERR_ALIGN
    assert call(ss=SS + 8) == binding.FP9_ERR_ALIGN
    assert call(x=P + 0x30004) == binding.FP9_ERR_ALIGN
    assert call(ws=WS + 16) == binding.FP9_ERR_ALIGN
    assert call(layer=_layer(topk=17)) == binding.FP9_ERR_SHAPE
    assert call(nxt=_layer(topk=17)) == binding.FP9_ERR_SHAPE       # the next layer is checked too
    assert call(nxt=_layer(w_router=P + 4)) == binding.FP9_ERR_ALIGN


def test_moe_forward_host_argument_checks(lib):
    # the host buffers are only dereferenced by the queued copies, which an
    # argument error never reaches
    xh = ctypes.create_string_buffer(4096)
    yh = ctypes.create_string_buffer(4096)
    L = _layer()

    def call(layer=L, x=xh, bsz=1, y=yh, ws=P, ws_bytes=1 << 30):
        return lib.fp9_moe_forward_host(ctypes.byref(layer) if layer is not None else None, x, bsz, y, ws,
                                        ws_bytes, None, None)
    assert call(layer=None) == binding.FP9_ERR_INVALID_ARG
    assert call(bsz=0) == binding.FP9_ERR_INVALID_ARG
    assert call(bsz=9) == binding.FP9_ERR_INVALID_ARG
    assert call(x=None) == binding.FP9_ERR_INVALID_ARG
    assert call(y=None) == binding.FP9_ERR_INVALID_ARG
    assert call(y=xh) == binding.FP9_ERR_INVALID_ARG          # y aliases x
    assert call(ws=None) == binding.FP9_ERR_INVALID_ARG
    assert call(ws=P + 16) == binding.FP9_ERR_ALIGN
    assert call(layer=_layer(topk=17)) == binding.FP9_ERR_SHAPE
    assert lib.fp9_moe_host_workspace_bytes(ctypes.byref(_layer(topk=17)), 1) == 0


def test_dense_and_norm_argument_checks(lib):
    b = _bank(2, 64, 256)
    assert lib.fp9_dense_ffn(ctypes.byref(b), P, 1, P + 4096, P, 1 << 20, None, None) == binding.FP9_ERR_SHAPE
    b = _bank(1, 64, 256)
    assert lib.fp9_dense_ffn(ctypes.byref(b), P, 1, P, P, 1 << 20, None, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_residual_rmsnorm(P, None, P, 1, 6, ctypes.c_float(1e-6), None) == binding.FP9_ERR_SHAPE
    assert lib.fp9_residual_rmsnorm(P, None, P, 0, 8, ctypes.c_float(1e-6), None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_residual_rmsnorm(P + 4, None, P, 1, 8, ctypes.c_float(1e-6), None) == binding.FP9_ERR_ALIGN
    assert lib.fp9_selftest_timeout(P, 1 << 20, None, 100, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_prefill_selftest_timeout(P, 1 << 20, None, 100, None) == binding.FP9_ERR_INVALID_ARG
    assert lib.fp9_prefill_selftest_timeout(P, 1 << 16, P, 100, None) == binding.FP9_ERR_WORKSPACE
    assert lib.fp9_prefill_selftest_timeout(P + 16, 1 << 20, P, 100, None) == binding.FP9_ERR_ALIGN
    assert lib.fp9_prefill_selftest_timeout(P, 1 << 20, P, 0, None) == binding.FP9_ERR_INVALID_ARG


def test_prefill_argument_checks(lib):
    b = _bank(2, 128, 512)

    def call(bank=b, k=0, x=P, m=4, y=P + 0x10000, ws=P + 0x20000, ws_bytes=1 << 30, precision=0):
        return lib.fp9_ffn_prefill(ctypes.byref(bank) if bank is not None else None, k, x, m, y, precision, ws,
                                   ws_bytes, None, None)

    need = lib.fp9_prefill_workspace_bytes(ctypes.byref(b), 4)
    assert need == 4 * 512 * 4 + 4 * 128 * 4     # x and h as two fp16 terms each, each 256-byte aligned
    assert call(precision=2) == binding.FP9_ERR_INVALID_ARG
    assert call(precision=-1) == binding.FP9_ERR_INVALID_ARG
    assert call(bank=None) == binding.FP9_ERR_INVALID_ARG
    assert call(k=2) == binding.FP9_ERR_INVALID_ARG
    assert call(k=-1) == binding.FP9_ERR_INVALID_ARG
    assert call(bank=_bank(2, 128, 384)) == binding.FP9_ERR_SHAPE        # hidden % 256
    assert call(bank=_bank(2, 100, 512)) == binding.FP9_ERR_SHAPE        # inter % 128
    assert call(bank=_bank(2, 128, 65536)) == binding.FP9_ERR_SHAPE      # > FP9_MAX_PREFILL_HIDDEN
    assert call(bank=_bank(2, 128, 512, base=P + 8)) == binding.FP9_ERR_ALIGN
    assert call(m=-1) == binding.FP9_ERR_INVALID_ARG
    assert call(m=binding.FP9_MAX_PREFILL_TOKENS + 1) == binding.FP9_ERR_INVALID_ARG
    assert call(m=0, x=None, y=None, ws=None) == binding.FP9_OK           # empty: no-op
    assert call(x=None) == binding.FP9_ERR_INVALID_ARG
    assert call(x=P + 4) == binding.FP9_ERR_ALIGN
    assert call(y=P + 8) == binding.FP9_ERR_ALIGN
    assert call(ws=P + 16) == binding.FP9_ERR_ALIGN
    assert call(ws_bytes=need - 1) == binding.FP9_ERR_WORKSPACE
    assert lib.fp9_prefill_workspace_bytes(ctypes.byref(_bank(2, 128, 384)), 4) == 0
    assert lib.fp9_prefill_workspace_bytes(ctypes.byref(b), -1) == 0


def test_moe_prefill_argument_checks(lib):
    def call(layer, m=16, x=P, y=P + 0x10000, ws=P + 0x20000, ws_bytes=1 << 40, precision=0):
        return lib.fp9_moe_prefill(ctypes.byref(layer), x, m, y, None, None, precision, ws, ws_bytes, None, None)

    L = _layer()
    need = lib.fp9_moe_prefill_workspace_bytes(ctypes.byref(L), 16)
    assert need > 16 * 3 * (8 * 256 + 4 * 128)
    assert lib.fp9_moe_prefill(None, P, 4, P, None, None, 0, P, 1, None, None) == binding.FP9_ERR_INVALID_ARG
    assert call(L, precision=3) == binding.FP9_ERR_INVALID_ARG
    assert call(_layer(hidden=384, routed=_bank(8, 128, 384), shared=_bank(1, 128, 384))) == binding.FP9_ERR_SHAPE
    assert call(_layer(inter=64, routed=_bank(8, 64, 256), shared=_bank(1, 64, 256))) == binding.FP9_ERR_SHAPE
    assert call(_layer(topk=17)) == binding.FP9_ERR_SHAPE
    assert call(L, m=-1) == binding.FP9_ERR_INVALID_ARG
    assert call(L, m=0, x=None, y=None, ws=None) == binding.FP9_OK
    assert call(L, x=P + 4) == binding.FP9_ERR_ALIGN
    assert call(L, ws=P + 16) == binding.FP9_ERR_ALIGN
    assert call(L, ws_bytes=need - 1) == binding.FP9_ERR_WORKSPACE
    assert lib.fp9_moe_prefill_workspace_bytes(ctypes.byref(_layer(topk=17)), 16) == 0
