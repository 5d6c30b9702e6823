"""GPU router (moe_route / moe_route_from_logits / moe_group_topk) against the
oracle: logits and ids bit-exact, weights within 1e-6 relative."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import CONFIGS, SCORE_SIGMOID_BIAS, SCORE_SOFTMAX
from tests.gpu_common import ensure_lib, host_bits, layer_inputs
from tests.test_oracle_router import page_sim_scores, placement_stats, _golden_rows

pytestmark = pytest.mark.gpu


def _route_gpu(cfg, x, w_r, bias):
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    ids, w, logits = moe.moe_route(cfg.shape(), x, w_r,
                                   bias if cfg.score == SCORE_SIGMOID_BIAS else None, ws,
                                   want_logits=True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return ids.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "few_large", "decode", "prefill"])
def test_route_bit_exact_full_size(name):
    ensure_lib()
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    ids, w, logits = _route_gpu(cfg, t["x"], t["w_r"], t["bias"])
    x_h, wr_h = host_bits(name, "x"), host_bits(name, "w_r")
    ref_logits = oracle.router_logits(x_h, wr_h)
    assert np.array_equal(logits.view(np.uint32), ref_logits.view(np.uint32))
    ref_ids, ref_w, _ = oracle.route_from_logits(ref_logits, t["bias"].cpu().numpy(), cfg.G,
                                                 cfg.topk_group, cfg.k, cfg.score,
                                                 cfg.bias_scale)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))
    # invariants: k distinct experts from at most topk_group groups, sum 1
    gs = cfg.E // cfg.G
    for r in range(0, cfg.T, max(1, cfg.T // 512)):
        assert len(set(ids[r].tolist())) == cfg.k
        assert len(set((ids[r] // gs).tolist())) <= cfg.topk_group
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= cfg.k * 2.0 ** -23)


@pytest.mark.parametrize("T,d,E,G,tg,k,score", [
    (37, 776, 3, 1, 1, 2, SCORE_SOFTMAX),        # small-E kernel, ragged d, E not % 8
    (5, 8, 1, 1, 1, 1, SCORE_SOFTMAX),           # one round, one expert
    (129, 7168, 8, 1, 1, 2, SCORE_SOFTMAX),      # small-E kernel, W_r 129 KB resident
    (300, 2048, 16, 4, 2, 4, SCORE_SIGMOID_BIAS),
    (64, 1024, 24, 3, 2, 3, SCORE_SIGMOID_BIAS),  # tiled 32 x 32 tiles
    (100, 512, 64, 8, 4, 6, SCORE_SIGMOID_BIAS),  # tiled 16 x 64 tiles
    (33, 264, 200, 8, 3, 5, SCORE_SIGMOID_BIAS),  # ragged d and E
    (1000, 4096, 32, 1, 1, 8, SCORE_SOFTMAX),
])
def test_route_bit_exact_shapes(T, d, E, G, tg, k, score):
    ensure_lib()
    import moe_inputs
    tns = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=T + d + E)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=score,
                 bias_scale=0.15)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    bias = tns["bias"] if score == SCORE_SIGMOID_BIAS else None
    ids, w, logits = moe.moe_route(shape, tns["x"], tns["w_r"], bias, ws, want_logits=True)
    torch.cuda.synchronize()
    from tests.gpu_common import bits
    ref_logits = oracle.router_logits(bits(tns["x"]), bits(tns["w_r"]))
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), ref_logits.view(np.uint32))
    ref_ids, ref_w, _ = oracle.route_from_logits(ref_logits, tns["bias"].cpu().numpy(), G, tg, k,
                                                 score, 0.15)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    gw = w.cpu().numpy()
    assert np.all(np.abs(gw - ref_w) <= 1e-6 * np.abs(ref_w))


def _rand_logits(T, E, seed, kind):
    g = np.random.default_rng(seed)
    if kind == "normal":
        return g.normal(0, 3, (T, E)).astype(np.float32)
    if kind == "ties":
        return (np.round(g.normal(0, 2, (T, E)) * 2) / 2).astype(np.float32)
    if kind == "const":
        return np.full((T, E), 0.25, dtype=np.float32)
    if kind == "saturated":
        return g.normal(0, 40, (T, E)).astype(np.float32)
    raise ValueError(kind)


@pytest.mark.parametrize("T,E,G,tg,k,score,kind", [
    (1, 256, 8, 4, 8, SCORE_SIGMOID_BIAS, "normal"),
    (1000, 256, 8, 4, 8, SCORE_SIGMOID_BIAS, "ties"),
    (333, 256, 8, 4, 8, SCORE_SIGMOID_BIAS, "const"),
    (500, 256, 8, 4, 8, SCORE_SIGMOID_BIAS, "saturated"),
    (257, 16, 4, 2, 2, SCORE_SIGMOID_BIAS, "ties"),
    (100, 48, 3, 2, 5, SCORE_SIGMOID_BIAS, "normal"),
    (129, 1024, 32, 7, 32, SCORE_SIGMOID_BIAS, "normal"),
    (64, 64, 8, 2, 16, SCORE_SIGMOID_BIAS, "ties"),       # k = all eligible experts
    (300, 8, 1, 1, 2, SCORE_SOFTMAX, "normal"),
    (300, 8, 1, 1, 2, SCORE_SOFTMAX, "ties"),
    (77, 96, 1, 1, 6, SCORE_SOFTMAX, "saturated"),
])
def test_route_from_logits_edge_cases(T, E, G, tg, k, score, kind):
    ensure_lib()
    logits = _rand_logits(T, E, T + E, kind)
    bias = np.random.default_rng(E).normal(0, 1, E).astype(np.float32)
    if kind == "ties":
        bias = np.round(bias * 4) / 4
    shape = dict(T=T, d=8, E=E, G=G, topk_group=tg, k=k, score=score, inter=64,
                 bias_scale=0.15)
    ids, w = moe.moe_route_from_logits(shape, torch.from_numpy(logits).cuda(),
                                       torch.from_numpy(bias).cuda())
    ref_ids, ref_w, _ = oracle.route_from_logits(logits, bias, G, tg, k, score, 0.15)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    got_w = w.cpu().numpy()
    assert np.all(np.abs(got_w - ref_w) <= 1e-6 * np.abs(ref_w))


def test_group_topk_reproduces_ep_deploy_simulation():
    ensure_lib()
    s32 = page_sim_scores().astype(np.float32)
    shape = dict(T=s32.shape[0], d=8, E=256, G=8, topk_group=4, k=8, inter=64,
                 score=SCORE_SIGMOID_BIAS, bias_scale=0.15)
    ids = moe.moe_group_topk(shape, torch.from_numpy(s32).cuda()).cpu().numpy()
    ref = oracle.select(s32.astype(np.float64), 8, 4, 8, True)
    assert np.array_equal(ids, ref)
    for nodes, gpus, place, ratio, ntok in _golden_rows():
        if place == "by_number":
            assert placement_stats(ids, 256, nodes, gpus) == (ratio, ntok)


# --------------------------------------------------------------------------
# Screened routing (moe_route without logits; d and E multiples of 64): ids
# equal to the fixed-order path's, weights bit for bit.
# --------------------------------------------------------------------------

def _screened_vs_fixed(shape, x, w_r, bias):
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    b = bias if shape["score"] == SCORE_SIGMOID_BIAS else None
    ids_s, w_s, _ = moe.moe_route(shape, x, w_r, b, ws)
    n_flag = moe.moe_route_screened_count(shape, ws)
    ids_f, w_f, logits = moe.moe_route(shape, x, w_r, b, ws, want_logits=True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ids_s, w_s = ids_s.cpu().numpy(), w_s.cpu().numpy()
    assert np.array_equal(ids_s, ids_f.cpu().numpy())
    assert np.array_equal(w_s.view(np.uint32), w_f.cpu().numpy().view(np.uint32))
    return ids_s, w_s, logits.cpu().numpy(), n_flag


@pytest.mark.parametrize("T,d,E,G,tg,k,score", [
    (300, 512, 64, 1, 1, 6, SCORE_SIGMOID_BIAS),
    (257, 1024, 128, 4, 2, 8, SCORE_SIGMOID_BIAS),
    (1000, 256, 256, 8, 4, 8, SCORE_SIGMOID_BIAS),
    (64, 7168, 256, 8, 4, 8, SCORE_SIGMOID_BIAS),
    (500, 512, 128, 1, 1, 4, SCORE_SOFTMAX),
    (33, 128, 1024, 32, 8, 32, SCORE_SIGMOID_BIAS),   # 32 experts per lane, k = 32
    (700, 1024, 256, 8, 3, 6, SCORE_SOFTMAX),          # softmax with groups (margin on logits)
    (1, 64, 64, 2, 1, 1, SCORE_SIGMOID_BIAS),
    (4100, 2048, 192, 3, 2, 8, SCORE_SIGMOID_BIAS),   # 33 m-tiles, ragged last tile
])
def test_screened_route_matches_oracle(T, d, E, G, tg, k, score):
    ensure_lib()
    import moe_inputs
    from tests.gpu_common import bits
    tns = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=3 * T + d + E)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=score,
                 bias_scale=0.15)
    ids, w, logits, n_flag = _screened_vs_fixed(shape, tns["x"], tns["w_r"], tns["bias"])
    assert 0 <= n_flag <= T
    ref_logits = oracle.router_logits(bits(tns["x"]), bits(tns["w_r"]))
    assert np.array_equal(logits.view(np.uint32), ref_logits.view(np.uint32))
    ref_ids, ref_w, _ = oracle.route_from_logits(ref_logits, tns["bias"].cpu().numpy(), G, tg, k,
                                                 score, 0.15)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))


def test_screened_route_all_ties_take_the_fixed_order_path():
    # zero router weight and bias: every score ties, no token is screened
    ensure_lib()
    T, d, E, G, tg, k = 200, 256, 128, 8, 3, 6
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    w_r = torch.zeros(d, E, dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    ids, w, _, n_flag = _screened_vs_fixed(shape, x, w_r, bias)
    assert n_flag == T
    # ties go to the lower group, then the lower expert; equal weights
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    _, ref_w, _ = oracle.route_from_logits(np.zeros((T, E), np.float32), np.zeros(E), G, tg, k,
                                           SCORE_SIGMOID_BIAS, 0.15)
    assert np.array_equal(w, ref_w)


def test_screened_route_duplicate_experts_tie_exactly():
    # experts 2j and 2j+1 share a weight column: exact ties in every token;
    # the pair split at the selection boundary is flagged, pairs inside keep
    # lower index first
    ensure_lib()
    from tests.gpu_common import bits
    T, d, E, G, tg, k = 512, 1024, 64, 4, 2, 5
    g = torch.Generator().manual_seed(11)
    half = (torch.randn(d, E // 2, generator=g) * 0.05).to(torch.bfloat16)
    w_r = half.repeat_interleave(2, dim=1).contiguous()
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    bias = torch.zeros(E, dtype=torch.float32)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    ids, w, _, n_flag = _screened_vs_fixed(shape, x.cuda(), w_r.cuda(), bias.cuda())
    assert n_flag == T   # k odd: the k-th and (k+1)-th experts always tie
    ref_ids, ref_w, _ = oracle.route(bits(x), bits(w_r), bias.numpy(), G, tg, k,
                                     SCORE_SIGMOID_BIAS)
    assert np.array_equal(ids, ref_ids)
    k2 = 4
    shape["k"] = k2
    ids, w, _, n_flag = _screened_vs_fixed(shape, x.cuda(), w_r.cuda(), bias.cuda())
    assert n_flag < T
    ref_ids, ref_w, _ = oracle.route(bits(x), bits(w_r), bias.numpy(), G, tg, k2,
                                     SCORE_SIGMOID_BIAS)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_screened_route_full_size(name):
    ensure_lib()
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    ids, w, logits, n_flag = _screened_vs_fixed(cfg.shape(), t["x"], t["w_r"], t["bias"])
    # the fixed-order path itself is pinned to the oracle in
    # test_route_bit_exact_full_size; the screen sends a small share back
    assert 0 <= n_flag < cfg.T // 5


def test_screened_count_is_minus_one_when_not_screened():
    ensure_lib()
    import moe_inputs
    # E = 16 (not a multiple of 64): the fixed-order path
    tns = moe_inputs.make_tensors_for_shape(64, 256, 16, 64, device="cuda", seed=2)
    shape = dict(T=64, d=256, E=16, G=4, topk_group=2, k=2, inter=64,
                 score=SCORE_SIGMOID_BIAS, bias_scale=0.15)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    moe.moe_route(shape, tns["x"], tns["w_r"], tns["bias"], ws)
    assert moe.moe_route_screened_count(shape, ws) == -1
