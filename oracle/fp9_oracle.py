"""fp9 FFN/MoE decode step: the CPU oracle (test infrastructure only).

Plain float64 numpy restatement of every step on the GPU hot path, written so
that each line can be checked against its source by eye. It shares no code,
table or constant generator with the CUDA library, and neither imports the
other. Only the tests, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` may use it.

Sources (the pages this method comes from):

[MEMOIR-FP9]  "一鸭三吃：我把评测鸭变成了满血 DeepSeek-V3.2 推理系统"
              (judgeduck.ai/duck-llm/zh/memoir.html), section
              "在只有 AVX2 的 N100 上，我先做出了单核 MLP fp9": the fp9 bit
              diagram (1 sign bit, 5 exponent bits with bias 15 as in IEEE
              fp16, 3 mantissa bits); storage as one body byte per weight plus
              a sign plane with 8 signs per byte; decoding by widening the body
              to 16 bits, shifting it left by 7 into a legal fp16 with the sign
              on top, then converting to fp32 with no exponent fix-up.
[MEMOIR-COMM] same page, section "真正难的不是把参数塞下，而是通信": the FFN is
              split tensor-parallel across nodes, whose f32 partial sums are
              then summed.
[MEMOIR-16]   same page, section "16 tok/s 之后": the MoE-forward breakdown,
              with the host-side reduce of the partial sums.
[MTP-9.2]     "第 9 章 MTP1 dual-lane overlap"
              (judgeduck.ai/duck-llm/zh/09-mtp1-dual-lane-overlap.html), §9.2:
              top_k = 8 experts per token; two tokens of a pair hit nearly
              disjoint expert sets.
[DS4-TP]      "ds4.c 学习笔记 — 张量并行"
              (ds4-learning.pages.dev/glossary/tensor-parallelism.html),
              section "形态一：Mac-to-Mac 张量并行": partial sums are f32 and are
              never quantised; a verify batch has at most 8 rows.

Readings where the pages are silent (each also listed in the design notes):

R1  Sign-bit order inside a sign byte: least significant bit first, i.e. the
    sign of column c sits in bit (c mod 8) of byte c // 8 of its row.
R2  Sign groups run along the contiguous (column) dimension of a row-major
    [rows, cols] matrix; cols must be a multiple of 8.
R3  Body byte layout: eeeeemmm (the 9-bit diagram with the sign bit removed).
R4  Encoding: round to nearest, ties to even mantissa, computed directly from
    the fp32 value (never through fp16); subnormals are kept; -0.0 keeps its
    sign. Magnitudes at or above 63488 (the midpoint between the largest
    finite value 61440 and 2**16), infinities and NaN are range errors: they
    are stored as the e=31 codes (+-Inf = body 0xF8, NaN = body 0xFC) and
    flagged.
R5  fp9 values carry no scale factor.
R6  e = 31 decodes like fp16: Inf when m = 0, NaN otherwise.
R7  Router (the pages only give top_k = 8): DeepSeek-V3-style sigmoid gate.
    Scores s = sigmoid(W_g x); experts form n_groups equal groups; a group's
    score is the sum of its two largest s (its only s when groups have one
    expert); the topk_groups best groups are kept (ties: lower group index);
    the topk best experts inside them are chosen (ties: lower expert id); the
    weights are s_i / sum(s_chosen) * route_scale. No score-correction bias.
R8  Shared experts are added with weight 1 (not multiplied by route_scale).
R9  W_down is stored transposed, as down_t = W_down^T of shape [I, H], so
    that each intermediate row's down weights are contiguous.
R10 Stack glue between layers: h <- h + MoE(RMSNorm(h)), eps 1e-6, unit gain.
R11 fp8 checkpoint conversion. The pages say that DeepSeek-V3 is published
    in fp8 ([MEMOIR-MEM]: about 688 GB on disk) and that its fp8 checkpoints
    use a 128x128 block-scale format ([QWEN]), and store fp9 weights without
    scales (R5); they give no formula. Plainest reading: each weight is an
    fp8 e4m3 byte (the variant without infinities: S.1111.111 is NaN; bias
    7; subnormals below 2**-6) times the fp32 scale of its 128x128 block of
    the [rows, cols] matrix (blocks at the right and bottom edges cover what
    is left); the product is exact in float64 (a 4-bit significand times a
    24-bit one) and is rounded once to fp9 as in R4, never through an fp32
    product, which could round it onto an fp9 midpoint first.

[MEMOIR-MEM]  "一鸭三吃" memoir, section "真正埋下伏笔的是内存；R1 之后，问题
              第一次被改写": the DeepSeek-V3 release format is fp8, about
              688 GB of weights on disk.
[QWEN]        same page, section "先用 Qwen3 练级，再让 Qwen3.5 充当高压试炼场":
              Qwen3's official fp8 checkpoints use the same 128x128
              block-scale format as DeepSeek-V3.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "FP9_INF_BODY", "FP9_NAN_BODY", "FP9_MAX", "FP9_OVERFLOW_THRESHOLD",
    "fp9_value", "fp9_encode", "fp9_pack", "fp9_unpack_signs", "fp9_decode",
    "router_scores", "route", "route_margin", "silu", "ffn", "moe", "dense_ffn",
    "rmsnorm", "stack", "FP8_BLOCK", "e4m3_value", "fp9_encode_exact", "fp8_block_to_fp9",
]

FP9_INF_BODY = 0xF8          # e = 31, m = 0
FP9_NAN_BODY = 0xFC          # e = 31, m = 4 (an fp16 quiet NaN once shifted)
FP9_MAX = 61440.0            # e = 30, m = 7: 2**15 * (1 + 7/8)
FP9_OVERFLOW_THRESHOLD = 63488.0   # midpoint of 61440 and 2**16 (R4)


# --------------------------------------------------------------------------
# The format
# --------------------------------------------------------------------------

def fp9_value(sign, body):
    """Value of fp9 codes, by the closed form of the bit diagram [MEMOIR-FP9].

    For exponent field e = body >> 3 and mantissa m = body & 7:
      e = 0        : 2**-14 * m / 8              (subnormal, as in fp16)
      1 <= e <= 30 : 2**(e - 15) * (1 + m / 8)
      e = 31       : Inf if m == 0 else NaN      (R6)
    and the sign bit negates. Returns float64.
    """
    sign = np.asarray(sign, dtype=np.int64)
    body = np.asarray(body, dtype=np.int64)
    e = body >> 3
    m = body & 7
    normal = np.ldexp(1.0 + m / 8.0, (e - 15).astype(np.int64))
    subnormal = np.ldexp(m / 8.0, -14)
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where(e == 31, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(sign != 0, -mag, mag)


_BLOCK = 1 << 20   # elements per block of the elementwise codec (memory only)


def _encode_block(x):
    sign = np.signbit(x).astype(np.uint8)
    a = np.abs(x.astype(np.float64))
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)

    _, k = np.frexp(a_f)                 # a = f * 2**k with f in [0.5, 1)
    e = np.maximum(k.astype(np.int64) - 1, -14)
    e = np.where(a_f == 0.0, -14, e)
    q = np.rint(a_f / np.ldexp(1.0, e - 3)).astype(np.int64)

    carry = q == 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)

    is_sub = (e == -14) & (q < 8)
    body = np.where(is_sub, q, ((e + 15) << 3) | (q - 8))

    overflow = finite & (e >= 16)
    range_error = ~finite | overflow
    body = np.where(overflow | np.isinf(a), FP9_INF_BODY, body)
    body = np.where(np.isnan(a), FP9_NAN_BODY, body)
    return sign, body.astype(np.uint8), range_error


def fp9_encode(x):
    """Encode fp32 values to fp9: returns (sign u8, body u8, range_error bool).

    Round to nearest, ties to even (R4), in exact float64 arithmetic: an fp32
    value and every fp9 value and midpoint are exact in float64.

    Steps: take the binade exponent e = floor(log2 |x|), clamped below at -14
    (the subnormal range shares the spacing of the lowest normal binade); the
    fp9 spacing there is 2**(e - 3); round |x| to a whole number q of spacings
    (numpy's rint rounds half to even); q < 8 with e = -14 is a subnormal;
    q = 16 carries into the next binade. Elements are independent; they are
    processed in blocks only to bound memory.
    """
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    sign = np.empty(flat.shape, np.uint8)
    body = np.empty(flat.shape, np.uint8)
    err = np.empty(flat.shape, bool)
    for i in range(0, flat.size, _BLOCK):
        sign[i:i + _BLOCK], body[i:i + _BLOCK], err[i:i + _BLOCK] = _encode_block(flat[i:i + _BLOCK])
    return sign.reshape(x.shape), body.reshape(x.shape), err.reshape(x.shape)


def fp9_encode_exact(x):
    """fp9_encode for float64 values that are exact as given (such as an
    fp8 value times an fp32 scale): the same rounding (R4), with no cast to
    fp32 first."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    sign = np.empty(flat.shape, np.uint8)
    body = np.empty(flat.shape, np.uint8)
    err = np.empty(flat.shape, bool)
    for i in range(0, flat.size, _BLOCK):
        sign[i:i + _BLOCK], body[i:i + _BLOCK], err[i:i + _BLOCK] = _encode_block(flat[i:i + _BLOCK])
    return sign.reshape(x.shape), body.reshape(x.shape), err.reshape(x.shape)


def _pack_signs(s):
    """Sign plane [rows, cols/8] from sign bits [rows, cols] (R1, R2)."""
    rows, cols = s.shape
    bits = s.reshape(rows, cols // 8, 8).astype(np.uint32)
    weights_of_bit = (1 << np.arange(8, dtype=np.uint32))
    return (bits * weights_of_bit).sum(axis=2).astype(np.uint8)


def fp9_pack(w):
    """Pack an fp32 matrix [rows, cols] into (body [rows, cols] u8,
    sign [rows, cols/8] u8, any_range_error) [MEMOIR-FP9], with the sign of
    column c in bit c % 8 of sign byte c // 8 (R1, R2)."""
    w = np.asarray(w, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % 8 != 0:
        raise ValueError("fp9_pack wants a 2-D matrix with cols % 8 == 0")
    s, body, err = fp9_encode(w)
    return body, _pack_signs(s), bool(err.any())


FP8_BLOCK = 128   # rows and columns of a scale block (R11)


def e4m3_value(code):
    """Value of fp8 e4m3 bytes as float64 (R11): sign bit 7, exponent bits
    6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal
    (m / 8 * 2**-6); S.1111.111 is NaN; there are no infinities."""
    code = np.asarray(code, dtype=np.int64)
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def fp8_block_to_fp9(w8, scale_inv):
    """Convert an fp8 block-scaled matrix to fp9 planes (R11).

    w8: e4m3 bytes [rows, cols] (cols % 8 == 0); scale_inv: fp32
    [ceil(rows / 128), ceil(cols / 128)], the scale of each 128x128 block.
    Returns (body [rows, cols] u8, sign [rows, cols / 8] u8, any_range_error).
    """
    w8 = np.asarray(w8, dtype=np.uint8)
    scale = np.asarray(scale_inv, dtype=np.float32).astype(np.float64)
    rows, cols = w8.shape
    if cols % 8 != 0:
        raise ValueError("fp8_block_to_fp9 wants cols % 8 == 0")
    nbr, nbc = -(-rows // FP8_BLOCK), -(-cols // FP8_BLOCK)
    if scale.shape != (nbr, nbc):
        raise ValueError("scale_inv must be [ceil(rows/128), ceil(cols/128)]")
    # the scale of each element: its block's, by the element's row and column
    per_elem = scale[(np.arange(rows) // FP8_BLOCK)[:, None], (np.arange(cols) // FP8_BLOCK)[None, :]]
    exact = e4m3_value(w8) * per_elem
    s, body, err = fp9_encode_exact(exact)
    return body, _pack_signs(s), bool(err.any())


def fp9_unpack_signs(sign, cols):
    """Sign bits [rows, cols] from a sign plane [rows, cols/8] (R1, R2)."""
    sign = np.asarray(sign, dtype=np.uint8)
    bit = (np.arange(cols) % 8).astype(np.uint8)
    byte = np.arange(cols) // 8
    return (sign[:, byte] >> bit[None, :]) & 1


_VALUE_OF_CODE = None


def fp9_decode(body, sign):
    """Decode packed planes to float64 [rows, cols] [MEMOIR-FP9].

    Each weight's 9-bit code (sign << 8 | body) is looked up in the table of
    fp9_value() over all 512 codes, i.e. the closed form per weight."""
    global _VALUE_OF_CODE
    if _VALUE_OF_CODE is None:
        codes = np.arange(512)
        _VALUE_OF_CODE = fp9_value(codes >> 8, codes & 0xFF)
    body = np.asarray(body, dtype=np.uint8)
    rows, cols = body.shape
    out = np.empty((rows, cols), np.float64)
    step = max(1, _BLOCK // max(cols, 1))
    for r in range(0, rows, step):
        s = fp9_unpack_signs(np.asarray(sign)[r:r + step], cols).astype(np.int16)
        out[r:r + step] = _VALUE_OF_CODE[(s << 8) | body[r:r + step]]
    return out


# --------------------------------------------------------------------------
# Router (R7): top_k = 8 per token in [MTP-9.2]; the rest is the
# DeepSeek-V3-style gate the workload names.
# --------------------------------------------------------------------------

def router_scores(x, w_router):
    """Sigmoid scores s = 1 / (1 + exp(-W_g x)) in float64, [T, E]."""
    logits = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    return 1.0 / (1.0 + np.exp(-logits))


def _group_scores(s_row, n_groups):
    g = s_row.reshape(n_groups, -1)
    if g.shape[1] == 1:
        return g[:, 0]
    top2 = np.sort(g, axis=1)[:, -2:]
    return top2.sum(axis=1)


def _rank(values):
    """Indices ordered by value descending, ties to the lower index."""
    idx = np.arange(len(values))
    return np.lexsort((idx, -np.asarray(values)))


def route(x, w_router, n_groups, topk_groups, topk, route_scale):
    """Group-limited top-k routing (R7). Returns (ids [T, k] int32 in
    descending score order, weights [T, k] float64)."""
    s = router_scores(x, w_router)
    T, E = s.shape
    ids = np.zeros((T, topk), np.int32)
    wts = np.zeros((T, topk), np.float64)
    gsize = E // n_groups
    for t in range(T):
        gs = _group_scores(s[t], n_groups)
        kept = _rank(gs)[:topk_groups]
        eligible = np.zeros(E, bool)
        for g in kept:
            eligible[g * gsize:(g + 1) * gsize] = True
        masked = np.where(eligible, s[t], -np.inf)
        chosen = _rank(masked)[:topk]
        ids[t] = chosen
        wts[t] = s[t, chosen] / s[t, chosen].sum() * route_scale
    return ids, wts


def route_margin(x, w_router, n_groups, topk_groups, topk):
    """Smallest score gap at any routing decision, per token (float64).

    The decisions are: which groups are kept (gap between the
    topk_groups-th and the next group score) and which experts are chosen
    (gap between the topk-th and the next eligible expert score). A token
    whose margin is tiny could be routed differently by an fp32 path.
    """
    s = router_scores(x, w_router)
    T, E = s.shape
    gsize = E // n_groups
    out = np.full(T, np.inf)
    for t in range(T):
        gs = _group_scores(s[t], n_groups)
        order = _rank(gs)
        if topk_groups < n_groups:
            out[t] = min(out[t], gs[order[topk_groups - 1]] - gs[order[topk_groups]])
        eligible = np.zeros(E, bool)
        for g in order[:topk_groups]:
            eligible[g * gsize:(g + 1) * gsize] = True
        el = np.sort(s[t][eligible])[::-1]
        if len(el) > topk:
            out[t] = min(out[t], el[topk - 1] - el[topk])
    return out


# --------------------------------------------------------------------------
# FFN / MoE
# --------------------------------------------------------------------------

def silu(z):
    """SiLU(z) = z / (1 + exp(-z)), float64."""
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def ffn(x, w_gate, w_up, w_down_t):
    """SwiGLU FFN on decoded float64 weights [MEMOIR-FP9] (the duck MLP).

    x [T, H]; w_gate, w_up, w_down_t [I, H] (w_down_t = W_down^T, R9).
    y = W_down (SiLU(W_gate x) * (W_up x)), returned as [T, H].
    """
    x = np.asarray(x, np.float64)
    g = x @ np.asarray(w_gate, np.float64).T
    u = x @ np.asarray(w_up, np.float64).T
    h = silu(g) * u
    return h @ np.asarray(w_down_t, np.float64)


def _decoded(planes):
    """planes = (gate_body, gate_sign, up_body, up_sign, down_body, down_sign)."""
    gb, gs, ub, us, db, ds = planes
    return fp9_decode(gb, gs), fp9_decode(ub, us), fp9_decode(db, ds)


def moe(x, w_router, routed, shared, n_groups, topk_groups, topk, route_scale,
        ids=None, weights=None):
    """One MoE layer on fp9 experts, float64.

    y[t] = sum_k w[t,k] * FFN_{ids[t,k]}(x[t]) + sum_s FFN_shared_s(x[t]) (R8).
    ``routed(e)`` and ``shared(s)`` return an expert's six packed planes;
    ``shared`` is a sequence. ``ids``/``weights`` override the router (used by
    the invariant tests). The sum over experts and over the intermediate
    dimension is the exact result that the split partial sums of
    [MEMOIR-COMM] / [MEMOIR-16] add up to.
    """
    x = np.asarray(x, np.float64)
    if ids is None:
        ids, weights = route(x, w_router, n_groups, topk_groups, topk, route_scale)
    y = np.zeros_like(x)
    cache = {}
    for t in range(x.shape[0]):
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            if e not in cache:
                cache[e] = _decoded(routed(e))
            y[t] += weights[t, k] * ffn(x[t:t + 1], *cache[e])[0]
    for planes in shared:
        wg, wu, wd = _decoded(planes)
        y += ffn(x, wg, wu, wd)
    return y


def dense_ffn(x, planes):
    """Dense SwiGLU FFN on one set of fp9 planes, float64."""
    return ffn(x, *_decoded(planes))


def rmsnorm(h, eps=1e-6):
    """h / sqrt(mean(h**2) + eps), unit gain, per row (R10)."""
    h = np.asarray(h, np.float64)
    return h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)


def stack(h, layers, eps=1e-6):
    """h <- h + MoE_l(RMSNorm(h)) for each layer (R10). ``layers`` is a
    sequence of dicts holding moe()'s keyword arguments except x."""
    h = np.asarray(h, np.float64).copy()
    for layer in layers:
        h = h + moe(rmsnorm(h, eps), **layer)
    return h
