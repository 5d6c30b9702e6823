"""Oracle pins for the capacity variant ("第十五章" section 4.3, "Capacity
Factor" and its overflow table): the capacity formula against the page's
worked example and exact rational arithmetic, the capacity dispatch against
a brute-force restatement and the uncapped dispatch, and the layer with
dropped assignments against the FFN of single rows."""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle
from moe_inputs import CONFIGS, bf16_bits, make_layer_tensors, random_ids


def test_capacity_page_example():
    # T = 5600 tokens, k = 16, E = 896: 100 assignments per expert on
    # average; c = 1.2 gives a capacity of about 120
    assert oracle.expert_capacity(5600, 16, 896, 1.0) == 100
    assert oracle.expert_capacity(5600, 16, 896, 1.2) == 120
    assert oracle.expert_capacity(5600, 16, 896, 1.5) == 150


@pytest.mark.parametrize("c", [1.0, 1.25, 1.5, 2.0, 0.5, 3.0])
def test_capacity_matches_exact_rational_ceiling(c):
    # c values exactly representable in binary: the double evaluation must
    # equal the exact ceiling
    g = np.random.default_rng(int(c * 100))
    for _ in range(300):
        T, k, E = int(g.integers(1, 20000)), int(g.integers(1, 17)), int(g.integers(1, 1025))
        want = math.ceil(Fraction(c) * T * k / E)
        assert oracle.expert_capacity(T, k, E, c) == want, (T, k, E, c)


def _brute_dispatch_capacity(ids, E, C, policy):
    T, k = ids.shape
    flat = ids.ravel()
    counts = np.bincount(flat, minlength=E)
    kept = np.minimum(counts, C)
    ovf = np.concatenate([[0], np.cumsum(counts - kept)])
    dest = np.full(T * k, -1, np.int64)
    src = np.full(E * C + T * k, -1, np.int64)
    for e in range(E):
        members = [a for a in range(T * k) if flat[a] == e]   # increasing a
        for r, a in enumerate(members):
            if r < C:
                row = e * C + r
            elif policy == 1:
                row = E * C + ovf[e] + (r - C)
            else:
                row = -1
            dest[a] = row
            if row >= 0:
                src[row] = a // k
    return counts, kept, ovf, dest, src


@pytest.mark.parametrize("T,k,E,C,skew", [
    (37, 2, 5, 3, 0.0), (64, 4, 8, 0, 1.0), (100, 8, 16, 40, 2.0), (257, 3, 7, 200, 0.5),
    (50, 6, 9, 1, 3.0)])
@pytest.mark.parametrize("policy", [0, 1])
def test_dispatch_capacity_matches_brute_force(T, k, E, C, skew, policy):
    ids = random_ids(T, k, E, seed=T + E + C, skew=skew).numpy()
    got = oracle.dispatch_capacity(ids, E, C, policy)
    want = _brute_dispatch_capacity(ids, E, C, policy)
    for name, g_, w_ in zip(["counts", "kept", "ovf_offsets", "dest", "src_row"], got, want):
        assert np.array_equal(g_, w_), name


def test_dispatch_capacity_without_overflow_is_the_plain_dispatch():
    ids = random_ids(300, 4, 12, seed=5, skew=1.5).numpy()
    E = 12
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    C = int(counts.max())
    for policy in (0, 1):
        c2, kept, ovf, dcap, srow = oracle.dispatch_capacity(ids, E, C, policy)
        assert np.array_equal(c2, counts) and np.array_equal(kept, counts)
        assert ovf[-1] == 0 and (dcap >= 0).all()
        e = ids.ravel()
        # same rank inside each expert, padded row base e*C instead of offsets[e]
        assert np.array_equal(dcap - e * C, dest - offsets[e])
        assert np.array_equal(srow[dcap], src[dest])


def test_layer_keep_mask_drops_exactly_the_masked_terms():
    cfg = CONFIGS["tiny"]
    t = make_layer_tensors(cfg, device="cpu")
    x, wr, wgu, wd = (bf16_bits(t[n]) for n in ("x", "w_r", "w_gate_up", "w_down"))
    bias = t["bias"].numpy()
    shape = cfg.shape()
    tokens = np.arange(0, cfg.T, 5, dtype=np.int32)
    y_all, ids, w = oracle.layer_tokens(x, wr, bias, wgu, wd, shape, tokens)
    keep1 = np.ones((tokens.size, cfg.k), np.uint8)
    y_keep1, _, _ = oracle.layer_tokens(x, wr, bias, wgu, wd, shape, tokens, keep=keep1)
    assert np.array_equal(y_all, y_keep1)        # second round: every term kept
    keep0 = np.zeros_like(keep1)
    y0, _, _ = oracle.layer_tokens(x, wr, bias, wgu, wd, shape, tokens, keep=keep0)
    assert not y0.any()                           # everything dropped
    # keep only j = 0: w0 * FFN_{e0}(x_t), from the row FFN on its own
    keep_first = keep0.copy()
    keep_first[:, 0] = 1
    y1, _, _ = oracle.layer_tokens(x, wr, bias, wgu, wd, shape, tokens, keep=keep_first)
    rows = oracle.expert_ffn_rows(x[tokens], ids[:, 0].astype(np.int32), wgu, wd)
    assert np.allclose(y1, w[:, :1].astype(np.float64) * rows.astype(np.float64), rtol=1e-12,
                       atol=1e-12)
