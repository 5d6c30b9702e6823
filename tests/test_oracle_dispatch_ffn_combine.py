"""Pins of the oracle's dispatch, expert FFN, combine and whole-layer
functions (no GPU)."""
import numpy as np
import pytest

import oracle
from moe_inputs import random_ids


def _bf16(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _f(bits):
    return oracle.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,skew", [(1, 1, 1, 0.0), (37, 2, 16, 0.0), (512, 8, 256, 2.0),
                                        (1000, 8, 256, 0.0), (300, 4, 7, 1.0)])
def test_dispatch_matches_sort_and_invariants(T, k, E, skew):
    ids = random_ids(T, k, E, seed=T + E, skew=skew).numpy()
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    flat = ids.reshape(-1)
    n = T * k
    # brute force: rows ordered by (expert, assignment index)
    order = np.lexsort((np.arange(n), flat))
    ref_dest = np.empty(n, dtype=np.int64)
    ref_dest[order] = np.arange(n)
    assert np.array_equal(dest, ref_dest)
    assert np.array_equal(src, order // k)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert counts.sum() == n
    assert offsets[0] == 0 and offsets[-1] == n
    assert np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(dest), np.arange(n))
    # each permuted row lies inside its expert's segment
    assert np.all((dest >= offsets[flat]) & (dest < offsets[flat + 1]))
    assert np.array_equal(src[dest], np.arange(n) // k)


def test_dispatch_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0, 5]], dtype=np.int32), 4)


# ---------------------------------------------------------------------------
# expert FFN
# ---------------------------------------------------------------------------

def _numpy_ffn(x, e, w_gu, w_down):
    xf, g_u, wd = _f(x), _f(w_gu), _f(w_down)
    inter = w_gu.shape[1] // 2
    out = np.empty((x.shape[0], w_down.shape[1]))
    for r in range(x.shape[0]):
        gu = g_u[e[r]] @ xf[r]
        g, u = gu[:inter], gu[inter:]
        h = g / (1.0 + np.exp(-g)) * u
        out[r] = wd[e[r]] @ h
    return out


def test_ffn_matches_numpy_float64():
    rng = np.random.default_rng(11)
    n, d, inter, E = 9, 256, 128, 3
    x = _bf16(rng.normal(0, 1, (n, d)))
    w_gu = _bf16(rng.normal(0, 0.02, (E, 2 * inter, d)))
    w_down = _bf16(rng.normal(0, 0.02, (E, d, inter)))
    e = rng.integers(0, E, n).astype(np.int32)
    got = oracle.expert_ffn_rows(x, e, w_gu, w_down)
    ref = _numpy_ffn(x, e, w_gu, w_down)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-7)


def test_ffn_closed_form_unit_weights():
    # gate row j = up row j = unit vector e_j, W_down = identity on the first
    # `inter` columns: g_j = u_j = x_j, so y_j = silu(x_j) * x_j for j < inter
    # and y_j = 0 beyond.
    rng = np.random.default_rng(12)
    n, d, inter = 5, 128, 64
    x = _bf16(rng.normal(0, 1.5, (n, d)))
    w_gu = np.zeros((1, 2 * inter, d), dtype=np.float32)
    w_down = np.zeros((1, d, inter), dtype=np.float32)
    for j in range(inter):
        w_gu[0, j, j] = 1.0
        w_gu[0, inter + j, j] = 1.0
        w_down[0, j, j] = 1.0
    y = oracle.expert_ffn_rows(x, np.zeros(n, dtype=np.int32), _bf16(w_gu), _bf16(w_down))
    xf = _f(x)[:, :inter]
    ref = xf * xf / (1.0 + np.exp(-xf))
    assert np.allclose(y[:, :inter], ref, rtol=1e-6, atol=1e-12)
    assert np.all(y[:, inter:] == 0)


def test_ffn_h_rounding_variant_is_bf16_of_h():
    rng = np.random.default_rng(13)
    n, d, inter = 4, 128, 64
    x = _bf16(rng.normal(0, 1, (n, d)))
    w_gu = _bf16(rng.normal(0, 0.05, (2, 2 * inter, d)))
    w_down = _bf16(rng.normal(0, 0.05, (2, d, inter)))
    e = np.array([0, 1, 1, 0], dtype=np.int32)
    _, h = oracle.expert_ffn_rows(x, e, w_gu, w_down, return_h=True)
    _, hr = oracle.expert_ffn_rows(x, e, w_gu, w_down, round_h_bf16=True, return_h=True)
    assert np.array_equal(hr, oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(h)))


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------

def test_combine_identity_experts_return_x():
    rng = np.random.default_rng(14)
    T, k, E, d = 50, 4, 8, 64
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    ids = random_ids(T, k, E, seed=3).numpy()
    _, _, dest, src = oracle.dispatch(ids, E)
    y_perm = x[src]  # identity experts
    w = rng.random((T, k)).astype(np.float32) + 0.1
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    y = oracle.combine(y_perm, dest, w, T, k)
    assert np.allclose(y, x, rtol=4e-7, atol=0)


def test_combine_one_hot_selects_expert_output():
    rng = np.random.default_rng(15)
    T, k, d = 20, 3, 16
    y_perm = rng.normal(0, 1, (T * k, d)).astype(np.float32)
    dest = rng.permutation(T * k).astype(np.int32)
    w = np.zeros((T, k), dtype=np.float32)
    pick = rng.integers(0, k, T)
    w[np.arange(T), pick] = 1.0
    y = oracle.combine(y_perm, dest, w, T, k)
    ref = y_perm[dest.reshape(T, k)[np.arange(T), pick]]
    assert np.array_equal(y, ref.astype(np.float64))


# ---------------------------------------------------------------------------
# whole layer for token subsets
# ---------------------------------------------------------------------------

def test_layer_tokens_equals_stage_composition():
    rng = np.random.default_rng(16)
    T, d, E, G, tg, k, inter = 24, 256, 16, 4, 2, 2, 128
    x = _bf16(rng.normal(0, 1, (T, d)))
    w_r = _bf16(rng.normal(0, 0.02, (d, E)))
    bias = rng.normal(0, 1, E).astype(np.float32)
    w_gu = _bf16(rng.normal(0, 0.02, (E, 2 * inter, d)))
    w_down = _bf16(rng.normal(0, 0.02, (E, d, inter)))
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=inter,
                 score=oracle.SCORE_SIGMOID_BIAS, bias_scale=0.15)
    ids, w, _ = oracle.route(x, w_r, bias, G, tg, k, oracle.SCORE_SIGMOID_BIAS)
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    y_perm = oracle.expert_ffn_rows(x[src], row_e, w_gu, w_down)
    y = oracle.combine(y_perm, dest, w, T, k)
    toks = np.array([0, 5, 23, 11], dtype=np.int32)
    y_sub, ids_sub, w_sub = oracle.layer_tokens(x, w_r, bias, w_gu, w_down, shape, toks)
    assert np.array_equal(ids_sub, ids[toks])
    assert np.array_equal(w_sub, w[toks])
    assert np.allclose(y_sub, y[toks], rtol=1e-6, atol=1e-7)
