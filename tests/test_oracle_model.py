"""Pins for the oracle's router, FFN, MoE and stack, against independent
formulations: exhaustive subset search for the router, pure-Python loops
for the FFN/MoE on tiny layers, and invariants that a dropped term, a wrong
sign or index or a transposed operand would break."""

import itertools
import math

import numpy as np
import pytest

import oracle as O


def _rand_planes(rng, rows, cols, std=0.02, zero=False):
    w = np.zeros((rows, cols), np.float32) if zero else \
        (rng.standard_normal((rows, cols)) * std).astype(np.float32)
    body, sign, err = O.fp9_pack(w)
    assert not err
    return body, sign


def _rand_ffn(rng, inter, hidden, zero=False):
    g = _rand_planes(rng, inter, hidden, zero=zero)
    u = _rand_planes(rng, inter, hidden, zero=zero)
    d = _rand_planes(rng, inter, hidden, zero=zero)
    return (*g, *u, *d)


def _fp16_value(sign, body):
    return float(np.array([(body << 7) | (sign << 15)], np.uint16).view(np.float16)[0])


def _naive_matrix(body, sign):
    """Decoded matrix as nested lists, through the fp16 reading."""
    rows, cols = body.shape
    return [[_fp16_value((int(sign[r, c // 8]) >> (c % 8)) & 1, int(body[r, c]))
             for c in range(cols)] for r in range(rows)]


def _naive_ffn(x, planes):
    gb, gs, ub, us, db, ds = planes
    G, U, D = _naive_matrix(gb, gs), _naive_matrix(ub, us), _naive_matrix(db, ds)
    inter, hidden = len(G), len(G[0])
    y = [0.0] * hidden
    for i in range(inter):
        g = sum(G[i][c] * x[c] for c in range(hidden))
        u = sum(U[i][c] * x[c] for c in range(hidden))
        h = g / (1.0 + math.exp(-g)) * u
        for c in range(hidden):
            y[c] += D[i][c] * h            # W_down[c, i] = down_t[i, c]
    return y


# ---------------------------------------------------------------- router ----

def _brute_route(x, wr, n_groups, topk_groups, topk, scale):
    """Exhaustive search: the kept groups are the topk_groups-subset with
    the largest total group score (a group's score is the largest sum of
    two of its members); the chosen experts are the topk-subset of the kept
    groups' experts with the largest total score."""
    E = wr.shape[0]
    s = [1.0 / (1.0 + math.exp(-sum(float(wr[e, c]) * float(x[c]) for c in range(len(x)))))
         for e in range(E)]
    gsize = E // n_groups
    gscore = []
    for g in range(n_groups):
        mem = range(g * gsize, (g + 1) * gsize)
        if gsize == 1:
            gscore.append(s[g])
        else:
            gscore.append(max(s[a] + s[b] for a, b in itertools.combinations(mem, 2)))
    kept = max(itertools.combinations(range(n_groups), topk_groups),
               key=lambda gs: sum(gscore[g] for g in gs))
    elig = [e for g in kept for e in range(g * gsize, (g + 1) * gsize)]
    chosen = max(itertools.combinations(elig, topk), key=lambda es: sum(s[e] for e in es))
    chosen = sorted(chosen, key=lambda e: -s[e])
    tot = sum(s[e] for e in chosen)
    return chosen, [s[e] / tot * scale for e in chosen]


@pytest.mark.parametrize("E,ng,tg,k,scale", [(8, 1, 1, 2, 1.0), (16, 4, 2, 3, 2.5),
                                             (12, 3, 1, 2, 1.0), (16, 8, 3, 4, 1.5)])
def test_router_matches_exhaustive_search(E, ng, tg, k, scale):
    rng = np.random.default_rng(E * 100 + k)
    H = 24
    for trial in range(6):
        x = rng.standard_normal((1, H))
        wr = rng.standard_normal((E, H)) * 0.3
        ids, w = O.route(x, wr, ng, tg, k, scale)
        bid, bw = _brute_route(x[0], wr, ng, tg, k, scale)
        assert list(ids[0]) == bid
        assert np.allclose(w[0], bw, rtol=1e-12, atol=0)
        assert abs(w[0].sum() - scale) < 1e-12


def test_router_without_group_limit_is_a_full_sort():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 40))
    wr = rng.standard_normal((32, 40)) * 0.2
    ids, w = O.route(x, wr, 1, 1, 8, 1.0)
    s = O.router_scores(x, wr)
    for t in range(3):
        assert list(ids[t]) == list(np.argsort(-s[t], kind="stable")[:8])


def test_router_ties_go_to_the_lower_index():
    # identical router rows give identical scores: lowest ids win, in order
    x = np.ones((1, 8))
    wr = np.zeros((8, 8))
    ids, w = O.route(x, wr, 1, 1, 3, 1.0)
    assert list(ids[0]) == [0, 1, 2]
    assert np.allclose(w[0], 1.0 / 3)
    # tied groups: the lower group is kept
    ids, _ = O.route(x, wr, 4, 1, 2, 1.0)
    assert list(ids[0]) == [0, 1]


def test_router_margin_is_the_smallest_decision_gap():
    # scores by construction: logits chosen so the 2nd/3rd gap is known
    E = 4
    logits = np.array([2.0, 1.0, 0.999, -1.0])
    x = np.ones((1, 1))
    wr = logits[:, None]
    m = O.route_margin(x, wr, 1, 1, 2)
    sig = 1.0 / (1.0 + np.exp(-logits))
    assert abs(m[0] - (sig[1] - sig[2])) < 1e-15
    # with groups of two, top-1 group: gap between the two group scores
    m = O.route_margin(x, wr, 2, 1, 2)
    gs = [sig[0] + sig[1], sig[2] + sig[3]]
    assert abs(m[0] - (gs[0] - gs[1])) < 1e-15


# ------------------------------------------------------------------- ffn ----

def test_ffn_matches_naive_loops():
    rng = np.random.default_rng(11)
    H, I, T = 16, 8, 3
    planes = _rand_ffn(rng, I, H)
    x = rng.standard_normal((T, H))
    y = O.dense_ffn(x, planes)
    for t in range(T):
        ref = _naive_ffn(list(x[t]), planes)
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)


def _tiny_layer(rng, H=16, I=8, E=8, ng=2, tg=1, k=2, n_shared=1, scale=1.0):
    experts = [_rand_ffn(rng, I, H) for _ in range(E)]
    shared = [_rand_ffn(rng, I, H) for _ in range(n_shared)]
    wr = rng.standard_normal((E, H)) * 0.3
    return dict(w_router=wr, routed=lambda e: experts[e], shared=shared,
                n_groups=ng, topk_groups=tg, topk=k, route_scale=scale), experts


def test_moe_matches_naive_loops():
    rng = np.random.default_rng(21)
    layer, experts = _tiny_layer(rng, n_shared=2, scale=2.5)
    x = rng.standard_normal((2, 16))
    y = O.moe(x, **layer)
    ids, w = _brute_ids(x, layer)
    for t in range(2):
        ref = [0.0] * 16
        for e, we in zip(ids[t], w[t]):
            f = _naive_ffn(list(x[t]), experts[e])
            ref = [a + we * b for a, b in zip(ref, f)]
        for sp in layer["shared"]:
            f = _naive_ffn(list(x[t]), sp)
            ref = [a + b for a, b in zip(ref, f)]
        assert np.allclose(y[t], ref, rtol=1e-11, atol=1e-14)


def _brute_ids(x, layer):
    ids, ws = [], []
    for t in range(x.shape[0]):
        i, w = _brute_route(x[t], layer["w_router"], layer["n_groups"],
                            layer["topk_groups"], layer["topk"], layer["route_scale"])
        ids.append(i)
        ws.append(w)
    return ids, ws


def test_moe_linearity_in_down_projection_is_exact():
    rng = np.random.default_rng(31)
    layer, experts = _tiny_layer(rng)
    x = rng.standard_normal((2, 16))
    y = O.moe(x, **layer)

    def doubled(p):
        d = O.fp9_decode(p[4], p[5]) * 2.0
        b, s, err = O.fp9_pack(d.astype(np.float32))
        assert not err
        return (*p[:4], b, s)

    exp2 = [doubled(p) for p in experts]
    layer2 = dict(layer, routed=lambda e: exp2[e], shared=[doubled(p) for p in layer["shared"]])
    assert np.array_equal(O.moe(x, **layer2), 2.0 * y)


def test_moe_routing_weight_scales_its_expert_term():
    rng = np.random.default_rng(41)
    layer, experts = _tiny_layer(rng)
    x = rng.standard_normal((1, 16))
    ids, w = O.route(x, layer["w_router"], 2, 1, 2, 1.0)
    base = O.moe(x, ids=ids, weights=w, **layer)
    w2 = w.copy()
    w2[0, 1] *= 3.0
    bumped = O.moe(x, ids=ids, weights=w2, **layer)
    term = w[0, 1] * O.dense_ffn(x, experts[ids[0, 1]])
    assert np.allclose(bumped - base, 2.0 * term, rtol=1e-10, atol=1e-14)


def test_moe_intermediate_permutation_invariance():
    rng = np.random.default_rng(51)
    layer, experts = _tiny_layer(rng)
    x = rng.standard_normal((2, 16))
    y = O.moe(x, **layer)
    perm = rng.permutation(8)
    pexp = [tuple(p[perm] for p in e) for e in experts]
    psh = [tuple(p[perm] for p in e) for e in layer["shared"]]
    y2 = O.moe(x, **dict(layer, routed=lambda e: pexp[e], shared=psh))
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-15)


def test_moe_expert_permutation_invariance():
    rng = np.random.default_rng(61)
    layer, experts = _tiny_layer(rng, E=8, ng=2, tg=1, k=2)
    x = rng.standard_normal((2, 16))
    y = O.moe(x, **layer)
    # swap the two groups and permute within each: routing follows the rows
    perm = np.array([5, 7, 4, 6, 1, 0, 3, 2])
    wr = layer["w_router"][perm]
    y2 = O.moe(x, **dict(layer, w_router=wr, routed=lambda e: experts[perm[e]]))
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-15)


def test_moe_zero_routed_experts_leave_the_shared_output():
    rng = np.random.default_rng(71)
    layer, _ = _tiny_layer(rng)
    zero = _rand_ffn(rng, 8, 16, zero=True)
    x = rng.standard_normal((2, 16))
    y = O.moe(x, **dict(layer, routed=lambda e: zero))
    ref = sum(O.dense_ffn(x, sp) for sp in layer["shared"])
    assert np.array_equal(y, ref)


def test_routing_weights_sum_to_scale():
    rng = np.random.default_rng(81)
    x = rng.standard_normal((8, 64))
    wr = rng.standard_normal((256, 64)) * 0.1
    ids, w = O.route(x, wr, 8, 4, 8, 2.5)
    assert np.allclose(w.sum(axis=1), 2.5, rtol=0, atol=1e-12)
    for t in range(8):
        assert len(set(ids[t])) == 8
        groups = set(int(e) // 32 for e in ids[t])
        assert len(groups) <= 4


# ----------------------------------------------------------------- stack ----

def test_rmsnorm_closed_form():
    h = np.array([[3.0, 4.0], [0.0, 0.0]])
    out = O.rmsnorm(h, 1e-6)
    assert np.allclose(out[0], h[0] / math.sqrt(12.5 + 1e-6), rtol=1e-15)
    assert np.array_equal(out[1], [0.0, 0.0])


def test_stack_with_zero_weights_is_identity_and_one_layer_matches_loops():
    rng = np.random.default_rng(91)
    layer0, _ = _tiny_layer(rng)
    zero = _rand_ffn(rng, 8, 16, zero=True)
    h = rng.standard_normal((2, 16))
    zl = dict(layer0, routed=lambda e: zero, shared=[zero])
    assert np.array_equal(O.stack(h, [zl, zl]), h)

    layer, experts = _tiny_layer(rng, n_shared=1)
    out = O.stack(h, [layer])
    for t in range(2):
        ms = sum(v * v for v in h[t]) / 16
        xn = [v / math.sqrt(ms + 1e-6) for v in h[t]]
        ids, w = _brute_route(np.array(xn), layer["w_router"], 2, 1, 2, 1.0)
        ref = list(h[t])
        for e, we in zip(ids, w):
            ref = [a + we * b for a, b in zip(ref, _naive_ffn(xn, experts[e]))]
        ref = [a + b for a, b in zip(ref, _naive_ffn(xn, layer["shared"][0]))]
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-14)
