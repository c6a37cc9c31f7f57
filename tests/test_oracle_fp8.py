"""Pins of the oracle's fp8 block-scale -> fp9 conversion (reading R11):
e4m3 decoding against torch's float8_e4m3fn conversion and hand-derived
values, single rounding of the exact product against a brute-force nearest
search, power-of-two scales converting exactly, double-rounding witnesses,
the 128x128 block indexing and the range cases. CPU only."""

import os
import struct

import numpy as np
import pytest
import torch

import oracle as O

HERE = os.path.dirname(__file__)


def _f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def _golden():
    rows = []
    with open(os.path.join(HERE, "golden", "fp8_to_fp9_worked_examples.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            f = line.split()
            rows.append((int(f[0], 16), int(f[1], 16), int(f[2]), int(f[3], 16), int(f[4])))
    return rows


# every finite fp9 value (sign, body) and its magnitude, for brute force
_CODES = [(s, b) for s in (0, 1) for b in range(0xF8)]
_MAGS = np.array([float(O.fp9_value(0, b)) for b in range(0xF8)])


def _brute_force(v):
    """Nearest finite fp9 to the exact value v (ties: even body), by search."""
    if np.isnan(v):
        return None
    a = abs(v)
    if a >= O.FP9_OVERFLOW_THRESHOLD:
        return "range"
    d = np.abs(_MAGS - a)
    best = np.flatnonzero(d == d.min())
    body = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return (1 if np.signbit(v) else 0), body


def test_e4m3_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_value(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(mine[ok]))


def test_golden_worked_examples():
    for code, sbits, sign, body, err in _golden():
        b, s, e = O.fp8_block_to_fp9(np.full((1, 8), code, np.uint8), np.array([[_f32(sbits)]], np.float32))
        assert int(b[0, 0]) == body, (hex(code), hex(sbits))
        assert int(s[0, 0] & 1) == sign, (hex(code), hex(sbits))
        assert bool(e) == bool(err), (hex(code), hex(sbits))


def test_power_of_two_scales_convert_exactly():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    x = O.e4m3_value(codes)
    for k in range(-8, 8):
        w8 = codes[None, : (len(codes) // 8) * 8]
        b, s, e = O.fp8_block_to_fp9(w8, np.full((1, 2), 2.0 ** k, np.float32))
        exact = x[: w8.shape[1]] * 2.0 ** k
        inside = (np.abs(exact) >= 2.0 ** -14) & (np.abs(exact) <= O.FP9_MAX)
        dec = O.fp9_decode(b, s)[0]
        assert np.array_equal(dec[inside], exact[inside]), k


def test_single_rounding_matches_brute_force():
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, size=(64, 128), dtype=np.uint8)
    for trial in range(12):
        scale = (np.exp2(rng.uniform(-20, 12)) * rng.choice([1.0, -1.0])).astype(np.float32).reshape(1, 1)
        b, s, _ = O.fp8_block_to_fp9(codes, scale)
        signs = O.fp9_unpack_signs(s, codes.shape[1])
        exact = O.e4m3_value(codes) * float(scale[0, 0])
        for idx in rng.integers(0, codes.size, size=300):
            r, c = divmod(int(idx), codes.shape[1])
            want = _brute_force(exact[r, c])
            if want is None:
                assert b[r, c] == O.FP9_NAN_BODY
            elif want == "range":
                assert b[r, c] == O.FP9_INF_BODY
            else:
                assert (int(signs[r, c]), int(b[r, c])) == want, (r, c, exact[r, c])


def test_double_rounding_witnesses_round_the_exact_product():
    found = 0
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
                exact = x * float(sc)
                if abs(float(np.float32(x) * sc)) != mid or abs(exact) == mid:
                    continue
                b, s, _ = O.fp8_block_to_fp9(np.full((1, 8), code, np.uint8), np.array([[sc]], np.float32))
                want = _brute_force(exact)
                assert (int(s[0, 0] & 1), int(b[0, 0])) == want
                found += 1
    assert found > 100  # the search does reach such cases


def test_block_indexing_follows_each_element():
    rng = np.random.default_rng(5)
    rows, cols = 200, 136
    codes = rng.integers(0, 0x7F, size=(rows, cols), dtype=np.uint8)  # positive, no NaN
    nbr, nbc = 2, 2
    scale = np.exp2(rng.integers(-6, 4, size=(nbr, nbc))).astype(np.float32)
    b, s, _ = O.fp8_block_to_fp9(codes, scale)
    dec = O.fp9_decode(b, s)
    for r in range(rows):
        for c in range(0, cols, 7):
            v = float(O.e4m3_value(codes[r, c])) * float(scale[r // 128, c // 128])
            if 2.0 ** -14 <= abs(v) <= O.FP9_MAX:
                assert dec[r, c] == v, (r, c)


def test_nan_and_range_cases():
    b, _, e = O.fp8_block_to_fp9(np.full((1, 8), 0x7F, np.uint8), np.array([[1.0]], np.float32))
    assert e and b[0, 0] == O.FP9_NAN_BODY
    # 61440 converts; 448 * 2^8 does not
    b, _, e = O.fp8_block_to_fp9(np.full((1, 8), 0x7E, np.uint8), np.array([[2.0 ** 7]], np.float32))
    assert not e
    b, _, e = O.fp8_block_to_fp9(np.full((1, 8), 0x7E, np.uint8), np.array([[2.0 ** 8]], np.float32))
    assert e and b[0, 0] == O.FP9_INF_BODY
    with pytest.raises(ValueError):
        O.fp8_block_to_fp9(np.zeros((4, 12), np.uint8), np.ones((1, 1), np.float32))
    with pytest.raises(ValueError):
        O.fp8_block_to_fp9(np.zeros((129, 8), np.uint8), np.ones((1, 1), np.float32))
