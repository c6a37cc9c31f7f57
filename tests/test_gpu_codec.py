"""GPU parity for fp9_pack / fp9_decode against the oracle: bit-exact bytes
and values, on random matrices, every rounding boundary, the special values
and ragged / empty shapes."""

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import binding

pytestmark = pytest.mark.gpu


def _gpu_pack(w_np):
    w = torch.from_numpy(np.ascontiguousarray(w_np, np.float32)).cuda()
    rows, cols = w.shape
    body = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    sign = torch.empty((rows, cols // 8), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_pack(w, body, sign, status)
    torch.cuda.synchronize()
    return body.cpu().numpy(), sign.cpu().numpy(), int(status.item())


def _boundaries():
    b = np.arange(0xF8)
    mags = np.append(O.fp9_value(np.zeros_like(b), b), 65536.0)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0)), mags[:-1].astype(np.float32)])
    vals = np.concatenate([vals, -vals])
    pad = (-len(vals)) % 64
    return np.concatenate([vals, np.zeros(pad, np.float32)]).reshape(-1, 64)


@pytest.mark.parametrize("shape", [(1, 8), (3, 24), (37, 136), (129, 7168), (2048, 256)])
def test_pack_matches_oracle_random(shape):
    rng = np.random.default_rng(shape[0] * 7 + shape[1])
    w = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    w.flat[:: max(1, w.size // 50)] *= 1e4          # some large magnitudes
    w.flat[1:: max(1, w.size // 40)] *= 1e-4         # some subnormal fp9
    body, sign, st = _gpu_pack(w)
    rb, rs, rerr = O.fp9_pack(w)
    assert st == 0 and not rerr
    assert np.array_equal(body, rb)
    assert np.array_equal(sign, rs)


def test_pack_matches_oracle_on_every_boundary():
    w = _boundaries()
    body, sign, st = _gpu_pack(w)
    rb, rs, rerr = O.fp9_pack(w)
    assert np.array_equal(body, rb)
    assert np.array_equal(sign, rs)
    assert rerr and st == binding.FP9_ERR_RANGE     # 63488 and above are in the set


def test_pack_special_values_and_status():
    w = np.zeros((2, 16), np.float32)
    w[0, :8] = [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-30, -1e-45, 61440.0]
    w[1, :8] = [63487.996, 63488.0, -70000.0, 2.0 ** -18, 3 * 2.0 ** -18, 2.0 ** -14, -1.0625, 1.9375]
    body, sign, st = _gpu_pack(w)
    rb, rs, rerr = O.fp9_pack(w)
    assert np.array_equal(body, rb) and np.array_equal(sign, rs)
    assert st == binding.FP9_ERR_RANGE
    ok = np.full((1, 8), 0.5, np.float32)
    assert _gpu_pack(ok)[2] == 0


def test_pack_empty_and_bad_shape():
    e = torch.empty((0, 16), device="cuda")
    binding.fp9_pack(e, torch.empty((0, 16), dtype=torch.uint8, device="cuda"),
                     torch.empty((0, 2), dtype=torch.uint8, device="cuda"))
    bad = torch.zeros((2, 12), device="cuda")
    with pytest.raises(binding.Fp9Error) as ei:
        binding.fp9_pack(bad, torch.empty((2, 12), dtype=torch.uint8, device="cuda"),
                         torch.empty((2, 2), dtype=torch.uint8, device="cuda"))
    assert ei.value.code == binding.FP9_ERR_SHAPE


def _gpu_decode(body, sign):
    b = torch.from_numpy(body).cuda()
    s = torch.from_numpy(sign).cuda()
    out = torch.empty(body.shape, dtype=torch.float32, device="cuda")
    binding.fp9_decode(b, s, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_decode_all_codes_bit_exact():
    # every (sign, body) pair at every column position of a sign byte
    rng = np.random.default_rng(0)
    body = np.tile(np.arange(256, dtype=np.uint8), 16).reshape(64, 64)
    sign = rng.integers(0, 256, (64, 8)).astype(np.uint8)
    got = _gpu_decode(body, sign)
    ref = O.fp9_decode(body, sign)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("shape", [(1, 8), (5, 40), (300, 7168)])
def test_decode_random_planes(shape):
    rng = np.random.default_rng(shape[1])
    body = rng.integers(0, 0xF8, shape).astype(np.uint8)
    sign = rng.integers(0, 256, (shape[0], shape[1] // 8)).astype(np.uint8)
    got = _gpu_decode(body, sign)
    ref = O.fp9_decode(body, sign).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_pack_then_decode_roundtrip_on_gpu_matches_oracle():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    body, sign, _ = _gpu_pack(w)
    got = _gpu_decode(body, sign)
    rb, rs, _ = O.fp9_pack(w)
    assert np.array_equal(got, O.fp9_decode(rb, rs).astype(np.float32))
