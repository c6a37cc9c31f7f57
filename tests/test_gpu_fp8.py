"""GPU parity for fp9_from_fp8 (fp8 e4m3 block-scale checkpoint -> fp9)
against the oracle: bit-exact body and sign planes, the range status, on
random codes and scales, ragged shapes (partial scale blocks, one group),
the hand-derived worked examples, products whose fp32 rounding lands on an
fp9 midpoint, and a full DeepSeek-V3 expert matrix. Ragged matrices take
the one-block-per-CTA kernel, matrices of whole blocks the persistent one."""

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import binding
from tests import test_oracle_fp8 as F8

pytestmark = pytest.mark.gpu


def _gpu(w8, scale):
    rows, cols = w8.shape
    body = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    sign = torch.empty((rows, cols // 8), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_from_fp8(torch.from_numpy(w8).cuda(), torch.from_numpy(scale).cuda(), body, sign, status)
    torch.cuda.synchronize()
    return body.cpu().numpy(), sign.cpu().numpy(), int(status.item())


def _check(w8, scale):
    b, s, st = _gpu(w8, scale)
    rb, rs, rerr = O.fp8_block_to_fp9(w8, scale)
    assert np.array_equal(b, rb)
    assert np.array_equal(s, rs)
    assert (st == binding.FP9_ERR_RANGE) == rerr and st in (0, binding.FP9_ERR_RANGE)


@pytest.mark.parametrize("rows,cols", [(1, 8), (128, 128), (200, 136), (129, 264), (300, 1024)])
def test_random_codes_and_block_scales(rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    w8 = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3C  # no NaN here (NaN is tested apart)
    nbr, nbc = -(-rows // 128), -(-cols // 128)
    scale = (np.exp2(rng.uniform(-14, 6, size=(nbr, nbc))) * rng.choice([1, -1], size=(nbr, nbc))).astype(np.float32)
    _check(w8, scale)


def test_worked_examples_and_midpoint_witnesses():
    for code, sbits, sign, body, err in F8._golden():
        w8 = np.full((1, 8), code, np.uint8)
        scale = np.array([[F8._f32(sbits)]], np.float32)
        b, s, st = _gpu(w8, scale)
        assert int(b[0, 0]) == body and int(s[0, 0] & 1) == sign, (hex(code), hex(sbits))
        assert (st == binding.FP9_ERR_RANGE) == bool(err)
    # every witness the oracle's search finds, as one matrix per scale
    for code in range(256):
        x = float(O.e4m3_value(code))
        if not np.isfinite(x) or x == 0:
            continue
        for mid in [1.0625 + 0.125 * j for j in range(8)]:
            s0 = np.float32(mid / abs(x))
            for step in (-2, -1, 1, 2):
                sc = s0
                for _ in range(abs(step)):
                    sc = np.nextafter(sc, np.float32(np.inf) if step > 0 else np.float32(-np.inf))
                if abs(float(np.float32(x) * sc)) != mid or abs(x * float(sc)) == mid:
                    continue
                _check(np.full((1, 8), code, np.uint8), np.array([[sc]], np.float32))


def test_nan_and_overflow_set_the_range_status():
    b, _, st = _gpu(np.full((1, 8), 0x7F, np.uint8), np.array([[1.0]], np.float32))
    assert st == binding.FP9_ERR_RANGE and b[0, 0] == O.FP9_NAN_BODY
    b, _, st = _gpu(np.full((1, 8), 0x7E, np.uint8), np.array([[256.0]], np.float32))
    assert st == binding.FP9_ERR_RANGE and b[0, 0] == O.FP9_INF_BODY
    _, _, st = _gpu(np.full((1, 8), 0x7E, np.uint8), np.array([[128.0]], np.float32))
    assert st == 0


def test_every_code_at_many_scales():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)[:248]
    rng = np.random.default_rng(3)
    w8 = np.tile(codes, (64, 1))
    scale = np.exp2(rng.uniform(-18, 8, size=(1, 2))).astype(np.float32)
    for _ in range(6):
        scale = np.exp2(rng.uniform(-18, 8, size=(1, 2))).astype(np.float32)
        _check(w8, scale)


def test_full_dsv3_expert_matrix():
    rng = np.random.default_rng(17)
    rows, cols = 2048, 7168
    w8 = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3C
    # checkpoint-like scales: weight magnitudes around 1e-2 after scaling
    scale = (np.exp2(rng.uniform(-14, -10, size=(rows // 128, cols // 128)))).astype(np.float32)
    _check(w8, scale)


def _midpoint_witnesses():
    """(code, scale) pairs whose fp32 product is an fp9 midpoint while the
    exact product is not (the oracle's rounding is decided by the latter)."""
    out = []
    for code in range(256):
        x = float(O.e4m3_value(code))
        if not np.isfinite(x) or x == 0:
            continue
        for mid in [1.0625 + 0.125 * j for j in range(8)]:
            s0 = np.float32(mid / abs(x))
            for step in (-1, 1):
                sc = np.nextafter(s0, np.float32(np.inf) if step > 0 else np.float32(-np.inf))
                if abs(float(np.float32(x) * sc)) == mid and abs(x * float(sc)) != mid:
                    out.append((code, sc))
    return out


@pytest.mark.parametrize("case", ["random", "nan", "overflow", "midpoints"])
def test_whole_blocks(case):
    """Matrices of whole 128 x 128 blocks run the persistent kernel, whose
    CTAs walk several blocks (here 45): bit-exact planes and the range
    status without NaN codes, with a NaN code in two blocks, with one block
    whose products overflow, and with blocks whose scale puts the fp32
    product of one code on an fp9 midpoint."""
    rows, cols = 640, 1152
    rng = np.random.default_rng(["random", "nan", "overflow", "midpoints"].index(case) + 40)
    w8 = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3C
    scale = (np.exp2(rng.uniform(-14, 6, size=(5, 9))) * rng.choice([1, -1], size=(5, 9))).astype(np.float32)
    if case == "nan":
        w8[130, 700] = 0x7F
        w8[639, 5] = 0xFF
    elif case == "overflow":
        scale[2, 3] = np.float32(2.0 ** 14)  # 448 * 2^14 is past the fp9 range
    elif case == "midpoints":
        wit = _midpoint_witnesses()
        assert len(wit) >= 45
        pick = rng.choice(len(wit), size=45, replace=False)
        for k, i in enumerate(pick):
            code, sc = wit[i]
            by, bx = divmod(k, 9)
            blk = w8[by * 128:(by + 1) * 128, bx * 128:(bx + 1) * 128]
            blk[rng.random(blk.shape) < 0.5] = code
            scale[by, bx] = sc
    _check(w8, scale)


def test_whole_blocks_several_per_cta():
    # 32 x 56 = 1792 blocks: more than the persistent grid holds at once
    rng = np.random.default_rng(23)
    rows, cols = 4096, 7168
    w8 = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3C
    scale = (np.exp2(rng.uniform(-14, -10, size=(rows // 128, cols // 128))) *
             rng.choice([1, -1], size=(rows // 128, cols // 128))).astype(np.float32)
    _check(w8, scale)


@pytest.mark.parametrize("cols", [8, 16])
def test_more_block_rows_than_one_grid_pass(cols):
    # 65539 block rows: the grid holds 65535 of them, so the CTAs of the
    # first 4 block rows also convert the last 4 (the last one ragged)
    rows = 65538 * 128 + 40
    rng = np.random.default_rng(cols)
    w8 = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x3C
    scale = (np.exp2(rng.uniform(-14, 6, size=(-(-rows // 128), 1))) *
             rng.choice([1, -1], size=(-(-rows // 128), 1))).astype(np.float32)
    b, s, st = _gpu(w8, scale)
    assert st == 0
    for r0, r1 in ((0, 4 * 128), (65534 * 128, rows)):
        rb, rs, rerr = O.fp8_block_to_fp9(w8[r0:r1], scale[r0 // 128:-(-r1 // 128)])
        assert not rerr
        assert np.array_equal(b[r0:r1], rb)
        assert np.array_equal(s[r0:r1], rs)
