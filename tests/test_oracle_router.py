"""Pins of the oracle's router (no GPU).

Each test checks the oracle against something other than itself: values the
ep-deploy handbook page prints, an fp64 dot product within the fp32 error
bound, hand-derived results that only the fixed summation order produces,
libm/numpy exp within an ulp bound, brute-force enumeration and numpy's
stable sort.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ep_deploy_routing_sim.txt")


def _bf16(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, np.finfo(np.float32).tiny)))
    return 2.0 ** (e - 23)


# ---------------------------------------------------------------------------
# exp / sigmoid
# ---------------------------------------------------------------------------

def test_exp_within_two_ulp_of_fp64():
    rng = np.random.default_rng(1)
    y = np.concatenate([
        rng.uniform(-80, 80, 200000),
        rng.uniform(-1, 1, 50000),
        np.array([0.0, -0.0, 1.0, -1.0, math.log(2), -math.log(2), 0.5 * math.log(2),
                  80.0, -80.0, 1e-8, -1e-8]),
    ]).astype(np.float32)
    got = oracle.exp(y).astype(np.float64)
    ref = np.exp(y.astype(np.float64))
    err = np.abs(got - ref) / _ulp32(ref)
    assert err.max() <= 2.0, err.max()


def test_exp_exact_points_and_clamp():
    assert oracle.exp(np.float32(0.0))[()] == 1.0
    # clamped outside [-80, 80]
    assert oracle.exp(np.float32(1000.0))[()] == oracle.exp(np.float32(80.0))[()]
    assert oracle.exp(np.float32(-1000.0))[()] == oracle.exp(np.float32(-80.0))[()]
    assert np.isfinite(oracle.exp(np.float32(80.0))[()])
    assert oracle.exp(np.float32(-80.0))[()] > 0.0


def test_sigmoid_within_bound_of_fp64():
    rng = np.random.default_rng(2)
    l = rng.normal(0, 4, 100000).astype(np.float32)
    got = oracle.sigmoid(l).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    err = np.abs(got - ref) / _ulp32(ref)
    assert err.max() <= 4.0, err.max()
    assert oracle.sigmoid(np.float32(0.0))[()] == 0.5


# ---------------------------------------------------------------------------
# logits
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,d,E", [(7, 256, 16), (5, 7168, 8), (3, 776, 24), (2, 8, 3)])
def test_logits_within_fp32_bound_of_fp64(T, d, E):
    rng = np.random.default_rng(T * 1000 + d)
    x = _bf16(rng.normal(0, 1, (T, d)))
    w = _bf16(rng.normal(0, 0.02, (d, E)))
    got = oracle.router_logits(x, w).astype(np.float64)
    xf = oracle.bf16_bits_to_f32(x).astype(np.float64)
    wf = oracle.bf16_bits_to_f32(w).astype(np.float64)
    ref = xf @ wf
    mag = np.abs(xf) @ np.abs(wf)
    depth = math.ceil(d / 256) * 8 + 5  # longest chain of roundings
    u = 2.0 ** -24
    bound = depth * u / (1 - depth * u) * mag
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


def test_logits_integer_inputs_are_exact():
    rng = np.random.default_rng(3)
    T, d, E = 4, 512, 8
    x = _bf16(rng.integers(-8, 9, (T, d)))
    w = _bf16(rng.integers(-8, 9, (d, E)))
    got = oracle.router_logits(x, w)
    ref = oracle.bf16_bits_to_f32(x).astype(np.int64) @ oracle.bf16_bits_to_f32(w).astype(np.int64)
    assert np.array_equal(got.astype(np.int64), ref)


def _order_case(positions):
    """x has 2**24 at i=0 and 1.0 at the listed positions; w = 1 (E=1)."""
    d = 512
    x = np.zeros((1, d), dtype=np.float32)
    x[0, 0] = 2.0 ** 24
    for p in positions:
        x[0, p] = 1.0
    w = np.ones((d, 1), dtype=np.float32)
    return oracle.router_logits(_bf16(x), _bf16(w))[0, 0]


def test_logits_fixed_order_hand_derived():
    # Lane 0 owns i in [0,8) and [256,264); lane 1 owns [8,16) and [264,272);
    # lane l owns chunks c with c mod 32 == l.
    # (a) 1.0 at i=1,2 (lane 0) and i=8,9 (lane 1): lane 0 = (2^24+1)+1 = 2^24
    #     (ties to even), lane 1 = 2; butterfly adds them last: 2^24 + 2.
    #     A plain sequential sum over i would give 2^24.
    assert _order_case([1, 2, 8, 9]) == 2.0 ** 24 + 2
    # (b) lanes 1 and 3 hold 1.0 each (i=8, i=24): the xor butterfly first
    #     forms lane1+lane3 = 2 (offset 2), then 2^24 + 2.  Lane-order or
    #     adjacent-pair trees give 2^24.
    assert _order_case([8, 24]) == 2.0 ** 24 + 2
    # (c) lanes 1 and 2 (i=8, i=16): offset 2 forms 2^24+1 -> 2^24 and
    #     lane1+lane3 = 1; offset 1 gives 2^24 + 1 -> 2^24.
    assert _order_case([8, 16]) == 2.0 ** 24
    # (d) second round of the same lane: i=256 and i=257 belong to lane 0,
    #     added after 2^24 one at a time: 2^24.  With i=264,265 (lane 1): +2.
    assert _order_case([256, 257]) == 2.0 ** 24
    assert _order_case([264, 265]) == 2.0 ** 24 + 2


# ---------------------------------------------------------------------------
# group-limited selection
# ---------------------------------------------------------------------------

def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            n, g, red, place, ratio, nodes = line.split()
            rows.append((int(n), int(g), place, ratio, nodes))
    return rows


def page_sim_scores():
    """The ep-deploy page's simulated scores (its stated recipe)."""
    rng = np.random.default_rng(0)
    E = 256
    bias = rng.normal(0, 1.0, E)
    scores = rng.random((20000, E)) + 0.15 * bias
    return scores


def placement_stats(ids, E, nodes, gpus):
    load = np.bincount(ids.ravel(), minlength=E).astype(float)
    per = E // gpus
    gpu_load = [float(load[i * per:(i + 1) * per].sum()) for i in range(gpus)]
    ratio = max(gpu_load) / float(np.mean(gpu_load))
    node_of = (np.arange(E) // per) // (gpus // nodes)
    touched = [len(set(node_of[r].tolist())) for r in ids[:2000]]
    return f"{ratio:.2f}", f"{float(np.mean(touched)):.2f}"


def test_select_reproduces_ep_deploy_printed_simulation():
    ids = oracle.select(page_sim_scores(), G=8, topk_group=4, k=8, group_sum_f32=False)
    checked = 0
    for nodes, gpus, place, ratio, ntok in _golden_rows():
        if place != "by_number":
            continue
        got = placement_stats(ids, 256, nodes, gpus)
        assert got == (ratio, ntok), (nodes, gpus, got, ratio, ntok)
        checked += 1
    assert checked == 2


def test_select_fp32_scores_same_on_page_recipe():
    s = page_sim_scores()
    a = oracle.select(s, 8, 4, 8, False)
    b = oracle.select(s.astype(np.float32).astype(np.float64), 8, 4, 8, True)
    assert np.array_equal(a, b)


def _brute_force(s, G, tg, k):
    """Unique (group set, expert set) with the defining order property."""
    E = len(s)
    gs = E // G
    if G > 1:
        gsc = []
        for g in range(G):
            top2 = sorted(s[g * gs:(g + 1) * gs], reverse=True)[:2]
            v = top2[0] + top2[1] if gs >= 2 else top2[0]
            gsc.append(float(np.float32(v)))
        key_g = lambda g: (gsc[g], -g)  # noqa: E731
        kept = None
        for cand in itertools.combinations(range(G), tg):
            rest = [g for g in range(G) if g not in cand]
            if all(key_g(a) > key_g(b) for a in cand for b in rest):
                assert kept is None
                kept = set(cand)
        elig = [e for e in range(E) if e // gs in kept]
    else:
        elig = list(range(E))
    key_e = lambda e: (s[e], -e)  # noqa: E731
    chosen = None
    for cand in itertools.combinations(elig, k):
        rest = [e for e in elig if e not in cand]
        if all(key_e(a) > key_e(b) for a in cand for b in rest):
            assert chosen is None
            chosen = cand
    return sorted(chosen, key=lambda e: (-s[e], e))


@pytest.mark.parametrize("G,tg,k", [(4, 2, 2), (4, 1, 3), (4, 3, 4), (2, 1, 2), (1, 1, 3)])
def test_select_brute_force_small(G, tg, k):
    rng = np.random.default_rng(G * 100 + tg * 10 + k)
    E = 16
    for trial in range(60):
        s = rng.normal(0, 1, E).astype(np.float32)
        if trial % 3 == 1:
            s = np.round(s * 2) / 2  # many exact ties
        if trial % 3 == 2:
            s[:] = s[0]  # all equal
        ids = oracle.select(s[None, :].astype(np.float64), G, tg, k, True)[0]
        assert list(ids) == _brute_force(s.astype(np.float64), G, tg, k)


def test_select_single_group_is_stable_topk():
    rng = np.random.default_rng(5)
    s = np.round(rng.normal(0, 1, (200, 8)), 1)
    ids = oracle.select(s, 1, 1, 2, False)
    ref = np.argsort(-s, axis=1, kind="stable")[:, :2]
    assert np.array_equal(ids, ref)


def test_select_constant_scores_pick_lowest_indices():
    s = np.zeros((3, 256))
    ids = oracle.select(s, 8, 4, 8, True)
    assert np.array_equal(ids, np.tile(np.arange(8), (3, 1)))


def test_select_respects_group_limit():
    rng = np.random.default_rng(6)
    s = rng.normal(0, 1, (500, 256))
    ids = oracle.select(s, 8, 4, 8, False)
    groups = ids // 32
    for r in range(len(ids)):
        assert len(set(ids[r].tolist())) == 8
        assert len(set(groups[r].tolist())) <= 4


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

def test_sigmoid_route_weights():
    rng = np.random.default_rng(7)
    T, E = 300, 64
    logits = rng.normal(0, 2, (T, E)).astype(np.float32)
    bias = rng.normal(0, 1, E).astype(np.float32)
    ids, w, sel = oracle.route_from_logits(logits, bias, G=8, topk_group=4, k=6,
                                           score=oracle.SCORE_SIGMOID_BIAS)
    # selection score = sigmoid + 0.15 bias (fp32)
    sig = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    assert np.allclose(sel, sig + 0.15 * bias, rtol=0, atol=6e-7)
    # weights = sigmoid of the chosen experts, renormalised (bias excluded)
    chosen = np.take_along_axis(sig, ids, 1)
    ref = chosen / chosen.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=2e-6, atol=0)
    assert np.all(w > 0)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 6 * 2.0 ** -23)
    # ids are in descending selection-score order
    ss = np.take_along_axis(sel, ids, 1)
    assert np.all(np.diff(ss, axis=1) <= 0)


def test_softmax_route_weights():
    rng = np.random.default_rng(8)
    T, E, k = 400, 8, 2
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    ids, w, _ = oracle.route_from_logits(logits, None, G=1, topk_group=1, k=k,
                                         score=oracle.SCORE_SOFTMAX)
    l64 = logits.astype(np.float64)
    p = np.exp(l64 - l64.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref_ids = np.argsort(-p, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    pk = np.take_along_axis(p, ids, 1)
    assert np.allclose(w, pk / pk.sum(1, keepdims=True), rtol=2e-6, atol=0)
