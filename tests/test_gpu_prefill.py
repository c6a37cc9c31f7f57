"""GPU parity for fp9_ffn_prefill (the FFN over many tokens on the tensor
cores) against the oracle's exact FFN. The default precision (activations
as two fp16 terms, hi + lo) is held to the decode path's rule, max|gpu -
oracle| <= 2e-4 * max|oracle| per token row; the opt-in one-term fp16 mode
to the tolerance its operand rounding implies (support.check_prefill)."""

import numpy as np
import pytest
import torch

import oracle as O
from fp9_weight_expert_gb300 import FFNBank, Workspace, binding, synth
from tests import support

pytestmark = pytest.mark.gpu


def _bank(n, hidden, inter, base):
    """An n-FFN bank packed on the GPU, and the oracle's decoded weights of
    each FFN (packed by the oracle from the same fp32 draws)."""
    f = FFNBank(n, inter, hidden)
    dec = []
    for k in range(n):
        planes = []
        for m in range(3):
            w = synth.ffn_weight(None, inter, hidden, synth.seed_for(base, 0, synth.DENSE, k, m), "cuda")
            f.pack(k, m, w)
            body, sign, err = O.fp9_pack(w.cpu().numpy())
            assert not err
            planes.append(O.fp9_decode(body, sign))
        dec.append(tuple(planes))
    return f, dec


SPLIT, FP16 = binding.FP9_PREFILL_SPLIT, binding.FP9_PREFILL_FP16
PRECISIONS = pytest.mark.parametrize("precision", [SPLIT, FP16], ids=["split", "fp16"])


def _run(f, x, k=0, out=None, precision=SPLIT):
    y = torch.empty_like(x) if out is None else out
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.fp9_ffn_prefill(f, x, y, Workspace.for_prefill(f, x.shape[0]).tensor, k, status, precision=precision)
    torch.cuda.synchronize()
    return y, int(status.item())


def _check(y, x, dec, precision):
    """The rule of each precision against the oracle's exact FFN."""
    if precision == SPLIT:
        ref = O.ffn(x, *dec)
        err = support.max_rel_err(y, ref)
        assert err <= support.TOL, f"max rel err {err:.3e} > {support.TOL}"
        return err
    return support.check_prefill(y, x, *dec)


# m spans one partial tile, exact tiles, ragged tails and several CTA tiles;
# (512, 256, 38900) is large enough that the kernels take 256-token tiles
# (two TMEM accumulators per operand) with a ragged last tile.
@pytest.mark.parametrize("hidden,inter,m", [
    (256, 128, 1), (256, 128, 5), (256, 128, 128), (256, 128, 129), (512, 384, 300),
    (1024, 512, 1000), (768, 1280, 517), (512, 256, 38900)])
@PRECISIONS
def test_prefill_matches_oracle(hidden, inter, m, precision):
    f, dec = _bank(1, hidden, inter, base=hidden * 7 + inter)
    x = synth.tokens(m, hidden, synth.seed_for(21, 0, synth.TOKENS, m), "cuda")
    y, st = _run(f, x, precision=precision)
    assert st == 0
    _check(y.cpu().numpy(), x.cpu().numpy().astype(np.float64), dec[0], precision)


@PRECISIONS
def test_prefill_selects_the_ffn_of_a_bank(precision):
    f, dec = _bank(3, 512, 256, base=77)
    x = synth.tokens(200, 512, 3, "cuda")
    for k in (2, 0, 1):
        y, st = _run(f, x, k, precision=precision)
        assert st == 0
        _check(y.cpu().numpy(), x.cpu().numpy().astype(np.float64), dec[k], precision)


def _sampled_rows(m):
    rows = {0, 1, 127, 128, 255, 256, m - 1, m - 2, m // 2}
    rng = np.random.default_rng(m)
    rows |= set(int(r) for r in rng.choice(m, 23, replace=False))
    return sorted(r for r in rows if 0 <= r < m)


# the pages' long prompt (1481 tokens) through one DeepSeek-V3 expert and
# through the dense FFN, checked on sampled token rows (each row of y
# depends only on its own row of x)
@pytest.mark.parametrize("hidden,inter,m", [(7168, 2048, 1481), (7168, 18432, 1481)])
@PRECISIONS
def test_prefill_full_size_sampled_rows(hidden, inter, m, precision):
    f, dec = _bank(1, hidden, inter, base=inter)
    x = synth.tokens(m, hidden, synth.seed_for(22, 0, synth.TOKENS, m), "cuda")
    y, st = _run(f, x, precision=precision)
    assert st == 0
    rows = _sampled_rows(m)
    xs = x.cpu().numpy().astype(np.float64)[rows]
    _check(y.cpu().numpy()[rows], xs, dec[0], precision)
    assert np.isfinite(y.cpu().numpy()).all()


@PRECISIONS
def test_prefill_is_deterministic_and_in_place(precision):
    f, dec = _bank(1, 1024, 512, base=5)
    x = synth.tokens(700, 1024, 8, "cuda")
    y1, _ = _run(f, x, precision=precision)
    y2, _ = _run(f, x, precision=precision)
    assert torch.equal(y1, y2)
    xi = x.clone()
    y3, st = _run(f, xi, out=xi, precision=precision)     # y aliases x
    assert st == 0
    assert torch.equal(y3, y1)


@PRECISIONS
def test_prefill_flags_out_of_range_values(precision):
    f, _ = _bank(1, 256, 128, base=9)
    x = synth.tokens(64, 256, 4, "cuda")
    x[3, 17] = 70000.0                # fp16 overflow in the input
    _, st = _run(f, x, precision=precision)
    assert st == binding.FP9_ERR_RANGE
    # h = SiLU(g) * u overflows fp16: every weight 2, every x 100
    g = FFNBank(1, 128, 256)
    for m in range(3):
        g.pack(0, m, torch.full((128, 256), 2.0, device="cuda"))
    _, st = _run(g, torch.full((8, 256), 100.0, device="cuda"), precision=precision)
    assert st == binding.FP9_ERR_RANGE


def test_prefill_rejects_an_unknown_precision():
    f, _ = _bank(1, 256, 128, base=9)
    x = synth.tokens(4, 256, 4, "cuda")
    with pytest.raises(binding.Fp9Error) as e:
        _run(f, x, precision=2)
    assert e.value.code == binding.FP9_ERR_INVALID_ARG


def test_prefill_matches_decode_path_within_tolerance():
    """The tensor-core path and the decode-step path (fp9_dense_ffn, fp32
    activations) agree: within the decode rule for the default precision,
    within the one-term tolerance for the fp16 mode."""
    f, dec = _bank(1, 1024, 256, base=31)
    x = synth.tokens(8, 1024, 10, "cuda")
    yd = torch.empty_like(x)
    binding.fp9_dense_ffn(f, x, yd, Workspace.for_dense(f, 8).tensor)
    y, st = _run(f, x)
    assert st == 0
    assert support.max_rel_err(y.cpu().numpy(), yd.cpu().numpy()) <= support.TOL
    y16, st = _run(f, x, precision=FP16)
    assert st == 0
    fro, row = support.prefill_errors(y16.cpu().numpy(), yd.cpu().numpy())
    assert fro <= support.PREFILL_FRO and row <= support.PREFILL_ROW


def test_prefill_workspace_holds_the_down_parts_for_small_m():
    # small m splits the down GEMM's K: the workspace then also holds fp32
    # partial outputs, and one with room for x and h only is rejected before
    # anything runs; large m needs x and h only
    f = FFNBank(1, 1280, 768)
    xh = 4 * (768 + 1280)  # bytes per token of x and h as two fp16 terms each
    small = binding.prefill_workspace_bytes(f, 517)
    assert small >= 517 * xh + 2 * 517 * 768 * 4
    big = binding.prefill_workspace_bytes(f, 65536)
    assert big < 65536 * xh + 1024
    x = torch.zeros((517, 768), dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    short = torch.zeros(517 * xh + 1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Fp9Error) as e:
        binding.fp9_ffn_prefill(f, x, y, short, 0)
    assert e.value.code == binding.FP9_ERR_WORKSPACE
