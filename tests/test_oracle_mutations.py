"""Planted mistakes in the oracle (on the CPU, by monkeypatching) must make
its pins fail: a wrong sign, index, transposition, rounding rule or
selection rule is caught by at least one pin."""

import numpy as np
import pytest

import oracle
import oracle.fp9_oracle as OM
from tests import test_oracle_codec as C
from tests import test_oracle_model as M


def _patch(monkeypatch, name, fn):
    """Replaces an oracle function in its module and in the package namespace."""
    monkeypatch.setattr(OM, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _fails(fn):
    with pytest.raises(AssertionError):
        fn()


def test_wrong_silu_sign_is_caught(monkeypatch):
    _patch(monkeypatch, "silu", lambda z: np.asarray(z, np.float64) / (1.0 + np.exp(np.asarray(z, np.float64))))
    _fails(M.test_ffn_matches_naive_loops)


def test_transposed_down_projection_is_caught(monkeypatch):
    def bad_ffn(x, wg, wu, wd):
        x = np.asarray(x, np.float64)
        h = OM.silu(x @ np.asarray(wg, np.float64).T) * (x @ np.asarray(wu, np.float64).T)
        return h @ np.asarray(wd, np.float64)[:, ::-1]
    _patch(monkeypatch, "ffn", bad_ffn)
    _fails(M.test_ffn_matches_naive_loops)


def test_top1_group_score_is_caught(monkeypatch):
    monkeypatch.setattr(OM, "_group_scores", lambda s, n: s.reshape(n, -1).max(axis=1))
    _fails(lambda: M.test_router_matches_exhaustive_search(16, 4, 2, 3, 2.5))


def test_ties_to_higher_index_is_caught(monkeypatch):
    monkeypatch.setattr(OM, "_rank", lambda v: np.lexsort((-np.arange(len(v)), -np.asarray(v))))
    _fails(M.test_router_ties_go_to_the_lower_index)


def test_round_half_up_is_caught(monkeypatch):
    orig = np.rint
    monkeypatch.setattr(OM.np, "rint", lambda a: np.floor(np.asarray(a) + 0.5))
    try:
        _fails(C.test_encode_matches_brute_force_on_every_boundary)
    finally:
        monkeypatch.setattr(OM.np, "rint", orig)


def test_msb_first_sign_plane_is_caught(monkeypatch):
    def bad_pack(w):
        w = np.asarray(w, np.float32)
        rows, cols = w.shape
        s, body, err = OM.fp9_encode(w)
        bits = s.reshape(rows, cols // 8, 8).astype(np.uint32)
        sign = (bits * (1 << np.arange(7, -1, -1, dtype=np.uint32))).sum(axis=2).astype(np.uint8)
        return body, sign, bool(err.any())
    _patch(monkeypatch, "fp9_pack", bad_pack)
    _fails(C.test_pack_sign_plane_bit_order_and_bodies)


def test_weights_normalised_over_all_experts_is_caught(monkeypatch):
    orig = OM.route

    def bad_route(x, wr, ng, tg, k, scale):
        ids, w = orig(x, wr, ng, tg, k, scale)
        s = OM.router_scores(x, wr)
        return ids, np.take_along_axis(s, ids.astype(np.int64), axis=1) / s.sum(axis=1, keepdims=True) * scale
    _patch(monkeypatch, "route", bad_route)
    _fails(M.test_routing_weights_sum_to_scale)


# --- fp8 block-scale conversion (R11) ---------------------------------------

from tests import test_oracle_fp8 as F8  # noqa: E402


def test_wrong_e4m3_bias_is_caught(monkeypatch):
    good = OM.e4m3_value

    def bad(code):
        return good(code) / 2.0  # bias 8 instead of 7
    _patch(monkeypatch, "e4m3_value", bad)
    _fails(F8.test_e4m3_matches_torch_float8)


def test_rounding_through_fp32_product_is_caught(monkeypatch):
    good = OM.fp9_encode_exact
    _patch(monkeypatch, "fp9_encode_exact", lambda x: good(np.asarray(x, np.float64).astype(np.float32)))
    _fails(F8.test_double_rounding_witnesses_round_the_exact_product)
    _fails(F8.test_golden_worked_examples)


def test_transposed_block_index_is_caught(monkeypatch):
    def bad(w8, scale_inv):
        w8 = np.asarray(w8, np.uint8)
        scale = np.asarray(scale_inv, np.float32).astype(np.float64)
        rows, cols = w8.shape
        per = scale[(np.arange(cols) // OM.FP8_BLOCK)[None, :], (np.arange(rows) // OM.FP8_BLOCK)[:, None]]
        s, body, err = OM.fp9_encode_exact(OM.e4m3_value(w8) * per)
        return body, OM._pack_signs(s), bool(err.any())
    _patch(monkeypatch, "fp8_block_to_fp9", bad)
    _fails(F8.test_block_indexing_follows_each_element)
