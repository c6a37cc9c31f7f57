"""Pins the prefill tolerance (support.check_prefill) on the CPU: an fp16
emulation of the path's arithmetic (x and h rounded by numpy's float16
conversion, fp32 GEMMs) passes it, and plausible mistakes in that path
fail it. Nothing here runs the CUDA library."""

import numpy as np
import pytest

import oracle as O
from tests import support


def _weights(hidden, inter, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(3):
        w = (rng.standard_normal((inter, hidden)) * 0.02).astype(np.float32)
        body, sign, err = O.fp9_pack(w)
        assert not err
        out.append(O.fp9_decode(body, sign))
    return out


def _emulate(x, wg, wu, wd, h_round="fp16", drop_chunk=None, swap_gate_up=False):
    """The prefill path's arithmetic with numpy: fp16 operands, fp32 sums."""
    x16 = x.astype(np.float16).astype(np.float32)
    g = x16 @ wg.T.astype(np.float32)
    u = x16 @ wu.T.astype(np.float32)
    if drop_chunk is not None:
        c = slice(64 * drop_chunk, 64 * drop_chunk + 64)
        g = g - x16[:, c] @ wg[:, c].T.astype(np.float32)
    if swap_gate_up:
        g, u = u, g
    h = g / (1.0 + np.exp(-g)) * u
    if h_round == "fp16":
        hr = h.astype(np.float16).astype(np.float32)
    else:  # bf16: keep the top 16 bits, rounding to nearest even
        b = h.astype(np.float32).view(np.uint32)
        hr = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32).view(np.float32)
    return (hr @ wd.astype(np.float32)).astype(np.float64)


@pytest.mark.parametrize("hidden,inter,m", [(256, 128, 64), (1024, 512, 48)])
def test_emulated_path_is_within_tolerance(hidden, inter, m):
    wg, wu, wd = _weights(hidden, inter, hidden)
    x = np.random.default_rng(1).standard_normal((m, hidden))
    fro, row = support.check_prefill(_emulate(x, wg, wu, wd), x, wg, wu, wd)
    assert 1e-4 < fro < 5e-4      # the two fp16 roundings are visible, and small


@pytest.mark.parametrize("mistake", [dict(h_round="bf16"), dict(drop_chunk=1), dict(swap_gate_up=True)])
def test_plausible_mistakes_fail_the_tolerance(mistake):
    wg, wu, wd = _weights(256, 128, 3)
    x = np.random.default_rng(2).standard_normal((64, 256))
    with pytest.raises(AssertionError):
        support.check_prefill(_emulate(x, wg, wu, wd, **mistake), x, wg, wu, wd)


def test_single_wrong_element_fails_the_bound():
    wg, wu, wd = _weights(256, 128, 4)
    x = np.random.default_rng(3).standard_normal((64, 256))
    y = _emulate(x, wg, wu, wd)
    y[17, 200] += 0.5 * np.abs(y).max()
    with pytest.raises(AssertionError, match="element-wise"):
        support.check_prefill(y, x, wg, wu, wd)


def test_bound_is_tight_enough_at_small_sizes():
    """At hidden 256 the worst-case bound stays well below the output scale,
    so a wrong element of the size of a typical output is caught."""
    wg, wu, wd = _weights(256, 128, 5)
    x = np.random.default_rng(4).standard_normal((32, 256))
    y = O.ffn(x, wg, wu, wd)
    b = support.prefill_error_bound(x, wg, wu, wd)
    assert np.sqrt(np.mean(b ** 2)) < 0.2 * np.sqrt(np.mean(y ** 2))
