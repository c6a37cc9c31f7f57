"""Pins for the oracle's fp9 codec, against things other than the oracle.

- decode: all 512 codes against numpy's IEEE float16 reading of
  (body << 7 | sign << 15), which is how the fp9 section of the JudgeDuck
  memoir says the format decodes ("shift the body left by 7 into a legal
  fp16, put the sign on top, widen to fp32");
- encode: a brute-force nearest-value search over every finite fp9 value,
  ties to the even mantissa, on all rounding boundaries and random values;
- pack: hand-derived worked examples (tests/golden) and the sign-plane bit
  order.
"""

import os
import struct

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp9_worked_examples.txt")


def _all_codes():
    s = np.repeat(np.arange(2), 256).astype(np.uint8)
    b = np.tile(np.arange(256), 2).astype(np.uint8)
    return s, b


def test_decode_exhaustive_matches_fp16_reading():
    s, b = _all_codes()
    bits16 = (b.astype(np.uint16) << 7) | (s.astype(np.uint16) << 15)
    lib = bits16.view(np.float16).astype(np.float64)
    mine = O.fp9_value(s, b)
    assert np.array_equal(np.isnan(lib), np.isnan(mine))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], mine[ok])
    # signed zeros
    assert np.array_equal(np.signbit(lib[ok]), np.signbit(mine[ok]))


def test_decode_closed_form_spot_values():
    # (-1)^s 2^(e-15) (1 + m/8), subnormal 2^-14 m/8
    assert O.fp9_value(0, (15 << 3) | 0) == 1.0
    assert O.fp9_value(1, (16 << 3) | 4) == -3.0
    assert O.fp9_value(0, (30 << 3) | 7) == 61440.0
    assert O.fp9_value(0, 1) == 2.0 ** -17
    assert O.fp9_value(0, 7) == 7 * 2.0 ** -17
    assert np.isinf(O.fp9_value(0, 0xF8)) and np.isnan(O.fp9_value(0, 0xF9))


def _finite_magnitudes():
    b = np.arange(0xF8)          # e < 31
    return b, O.fp9_value(np.zeros_like(b), b)


def _brute_force_encode(x):
    """Nearest fp9 magnitude by exhaustive search; ties to even body; the
    virtual value 2^16 (even body 0xF8) stands for overflow."""
    bodies, mags = _finite_magnitudes()
    bodies = np.append(bodies, 0xF8)
    mags = np.append(mags, 65536.0)
    out_b = np.zeros(len(x), np.int64)
    out_err = np.zeros(len(x), bool)
    for i, v in enumerate(np.asarray(x, np.float32).astype(np.float64)):
        if not np.isfinite(v):
            out_b[i] = 0xFC if np.isnan(v) else 0xF8
            out_err[i] = True
            continue
        d = np.abs(mags - abs(v))
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = best[bodies[best] % 2 == 0]
        out_b[i] = bodies[best[0]]
        out_err[i] = out_b[i] == 0xF8
    return out_b, out_err


def _boundary_values():
    _, mags = _finite_magnitudes()
    mags = np.append(mags, 65536.0)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)   # exact in fp32
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    vals = np.concatenate([mids, up, dn, mags.astype(np.float32)])
    return np.concatenate([vals, -vals])


def test_encode_matches_brute_force_on_every_boundary():
    x = _boundary_values()
    b, err = _brute_force_encode(x)
    s_o, b_o, err_o = O.fp9_encode(x)
    assert np.array_equal(b_o.astype(np.int64), b)
    assert np.array_equal(err_o, err)
    assert np.array_equal(s_o, np.signbit(x).astype(np.uint8))


def test_encode_matches_brute_force_random():
    rng = np.random.default_rng(1234)
    logu = (2.0 ** rng.uniform(-30, 17, 3000)).astype(np.float32)
    gauss = (rng.standard_normal(3000) * 0.02).astype(np.float32)
    denorm = (rng.integers(1, 1 << 23, 200).astype(np.uint32)).view(np.float32)
    x = np.concatenate([logu, -logu, gauss, denorm, -denorm,
                        np.array([0.0, -0.0, np.inf, -np.inf, np.nan], np.float32)])
    b, err = _brute_force_encode(x)
    s_o, b_o, err_o = O.fp9_encode(x)
    assert np.array_equal(b_o.astype(np.int64), b)
    assert np.array_equal(err_o, err)


def test_encode_roundtrip_every_finite_code():
    s, b = _all_codes()
    finite = (b >> 3) < 31
    s, b = s[finite], b[finite]
    v = O.fp9_value(s, b).astype(np.float32)
    s2, b2, err = O.fp9_encode(v)
    assert not err.any()
    assert np.array_equal(s2, s) and np.array_equal(b2, b)


def test_encode_fp16_values_with_seven_zero_low_bits_are_exact():
    rng = np.random.default_rng(7)
    h = rng.integers(0, 1 << 16, 5000).astype(np.uint16) & np.uint16(0xFF80)
    h = h[((h >> 10) & 0x1F) != 0x1F]           # drop Inf/NaN
    v = h.view(np.float16).astype(np.float32)
    s, b, err = O.fp9_encode(v)
    assert not err.any()
    assert np.array_equal(b.astype(np.uint16), (h >> 7) & 0xFF)
    assert np.array_equal(s.astype(np.uint16), h >> 15)


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = line.split()
            rows.append((struct.unpack(">f", bytes.fromhex(p[0]))[0],
                         int(p[1]), int(p[2], 16), int(p[3])))
    return rows


def test_golden_worked_examples():
    rows = _golden_rows()
    assert len(rows) >= 20
    x = np.array([r[0] for r in rows], np.float32)
    s, b, err = O.fp9_encode(x)
    for i, (v, sign, body, e) in enumerate(rows):
        assert (int(s[i]), int(b[i]), int(err[i])) == (sign, body, e), (v, s[i], hex(b[i]))
    # and the brute force agrees with the hand derivations
    bb, berr = _brute_force_encode(x)
    assert [int(v) for v in bb] == [r[2] for r in rows]


def test_pack_sign_plane_bit_order_and_bodies():
    cols = 24
    w = np.full((3, cols), 1.0, np.float32)
    for c in range(cols):
        w[c % 3, c] = -1.0           # row r has negatives at columns c = r mod 3
    body, sign, err = O.fp9_pack(w)
    assert not err
    assert body.shape == (3, cols) and sign.shape == (3, cols // 8)
    assert (body == 0x78).all()
    for r in range(3):
        for c in range(cols):
            bit = (sign[r, c // 8] >> (c % 8)) & 1
            assert bit == (1 if c % 3 == r else 0)
    # LSB-first: a lone negative at column 0 sets bit 0, at column 7 bit 7
    w = np.ones((1, 8), np.float32)
    w[0, 0] = -2.0
    assert O.fp9_pack(w)[1][0, 0] == 0x01
    w = np.ones((1, 8), np.float32)
    w[0, 7] = -2.0
    assert O.fp9_pack(w)[1][0, 0] == 0x80


def test_pack_rejects_ragged_columns_and_flags_range():
    with pytest.raises(ValueError):
        O.fp9_pack(np.zeros((2, 12), np.float32))
    w = np.zeros((2, 8), np.float32)
    w[1, 3] = 70000.0
    body, sign, err = O.fp9_pack(w)
    assert err and body[1, 3] == 0xF8


def test_decode_inverts_pack_up_to_rounding():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((16, 64)) * 0.02).astype(np.float32)
    body, sign, _ = O.fp9_pack(w)
    d = O.fp9_decode(body, sign)
    # relative error of round-to-nearest with 3 mantissa bits is <= 2^-4
    # for normal values; subnormals are within half a spacing 2^-18
    err = np.abs(d - w.astype(np.float64))
    bound = np.maximum(np.abs(w) * 2.0 ** -4, 2.0 ** -18)
    assert (err <= bound).all()
    assert np.array_equal(np.signbit(d), np.signbit(w))
