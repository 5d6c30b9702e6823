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
# Screened routing (moe_route without logits; d and E multiples of 64): the
# tensor-core logits bound every score to an interval, the experts left open
# get fixed-order logits; ids equal to the fixed-order path's, weights bit
# for bit, for any finite input.
# --------------------------------------------------------------------------

def _screened_vs_fixed(shape, x, w_r, bias, ws=None):
    ws = ws or moe.Workspace(moe.moe_workspace_size(shape))
    b = bias if shape["score"] == SCORE_SIGMOID_BIAS else None
    ids_s, w_s, _ = moe.moe_route(shape, x, w_r, b, ws)
    n_ref = moe.moe_route_refined_count(shape, ws)
    ids_f, w_f, logits = moe.moe_route(shape, x, w_r, b, ws, want_logits=True)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ids_s, w_s = ids_s.cpu().numpy(), w_s.cpu().numpy()
    assert np.array_equal(ids_s, ids_f.cpu().numpy())
    assert np.array_equal(w_s.view(np.uint32), w_f.cpu().numpy().view(np.uint32))
    T, k, E = shape["T"], shape["k"], shape["E"]
    assert T * k <= n_ref <= T * E  # every selected expert is refined
    return ids_s, w_s, logits.cpu().numpy(), n_ref


@pytest.mark.parametrize("T,d,E,G,tg,k,score", [
    (300, 512, 64, 1, 1, 6, SCORE_SIGMOID_BIAS),
    (257, 1024, 128, 4, 2, 8, SCORE_SIGMOID_BIAS),
    (1000, 256, 256, 8, 4, 8, SCORE_SIGMOID_BIAS),
    (64, 7168, 256, 8, 4, 8, SCORE_SIGMOID_BIAS),
    (500, 512, 128, 1, 1, 4, SCORE_SOFTMAX),
    (33, 128, 1024, 32, 8, 32, SCORE_SIGMOID_BIAS),   # 32 experts per lane, k = 32
    (700, 1024, 256, 8, 3, 6, SCORE_SOFTMAX),          # softmax with groups (intervals on logits)
    (1, 64, 64, 2, 1, 1, SCORE_SIGMOID_BIAS),
    (4100, 2048, 192, 3, 2, 8, SCORE_SIGMOID_BIAS),   # 33 m-tiles, ragged last tile, E % 256 != 0
    (129, 16384, 320, 5, 2, 8, SCORE_SIGMOID_BIAS),   # largest d, 64-wide tiles
])
def test_screened_route_matches_oracle(T, d, E, G, tg, k, score):
    ensure_lib()
    import moe_inputs
    from tests.gpu_common import bits
    tns = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=3 * T + d + E)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=score,
                 bias_scale=0.15)
    ids, w, logits, n_ref = _screened_vs_fixed(shape, tns["x"], tns["w_r"], tns["bias"])
    ref_logits = oracle.router_logits(bits(tns["x"]), bits(tns["w_r"]))
    assert np.array_equal(logits.view(np.uint32), ref_logits.view(np.uint32))
    ref_ids, ref_w, _ = oracle.route_from_logits(ref_logits, tns["bias"].cpu().numpy(), G, tg, k,
                                                 score, 0.15)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))


@pytest.mark.parametrize("T,d,E,G,tg,k,score", [
    (8193, 1088, 64, 4, 2, 6, SCORE_SIGMOID_BIAS),   # ragged last tile, d % 128 == 64
    (9000, 2048, 256, 8, 4, 8, SCORE_SIGMOID_BIAS),
    (8200, 512, 128, 1, 1, 4, SCORE_SOFTMAX),
])
def test_screened_route_large_T(T, d, E, G, tg, k, score):
    # large token counts (the refinement's one-expert-per-warp form), ragged
    # T and d % 128 == 64: the same ids and weight bits as the fixed-order
    # path, and sampled tokens equal to the oracle's
    ensure_lib()
    import moe_inputs
    from tests.gpu_common import bits
    tns = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=T + 7 * d + E)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=score,
                 bias_scale=0.15)
    ids, w, _, n_ref = _screened_vs_fixed(shape, tns["x"], tns["w_r"], tns["bias"])
    rows = np.unique(np.concatenate([np.arange(0, T, max(1, T // 40)), [T - 1]]))
    xs = bits(tns["x"])[rows]
    ref_ids, ref_w, _ = oracle.route(xs, bits(tns["w_r"]), tns["bias"].cpu().numpy(), G, tg, k,
                                     score)
    assert np.array_equal(ids[rows], ref_ids)
    assert np.all(np.abs(w[rows] - ref_w) <= 1e-6 * np.abs(ref_w))


def test_screened_route_large_T_all_ties():
    # nearly every expert of every token refined, at a large token count
    ensure_lib()
    T, d, E, G, tg, k = 8192, 256, 128, 8, 3, 6
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    w_r = torch.zeros(d, E, dtype=torch.bfloat16, device="cuda")
    w_r[3, 5] = 1.0  # expert 5 wins where x[:, 3] > 0, else an all-tie
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    ids, w, _, n_ref = _screened_vs_fixed(shape, x, w_r, bias)
    assert n_ref > T * 100


def test_screened_route_all_ties_refine_everything():
    # zero router weight and bias: every score ties, so every interval
    # overlaps every other and all E experts of every token are refined
    ensure_lib()
    T, d, E, G, tg, k = 200, 256, 128, 8, 3, 6
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    w_r = torch.zeros(d, E, dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(E, dtype=torch.float32, device="cuda")
    ids, w, _, n_ref = _screened_vs_fixed(shape, x, w_r, bias)
    assert n_ref == T * E
    # ties go to the lower group, then the lower expert; equal weights
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    _, ref_w, _ = oracle.route_from_logits(np.zeros((T, E), np.float32), np.zeros(E), G, tg, k,
                                           SCORE_SIGMOID_BIAS, 0.15)
    assert np.array_equal(w, ref_w)


def test_screened_route_duplicate_experts_tie_exactly():
    # experts 2j and 2j+1 share a weight column: exact ties in every token;
    # with k odd the k-th and (k+1)-th experts tie, so both are refined and
    # the lower index wins
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
    ids, w, _, n_ref = _screened_vs_fixed(shape, x.cuda(), w_r.cuda(), bias.cuda())
    assert n_ref >= T * (k + 1)
    ref_ids, ref_w, _ = oracle.route(bits(x), bits(w_r), bias.numpy(), G, tg, k,
                                     SCORE_SIGMOID_BIAS)
    assert np.array_equal(ids, ref_ids)
    for k2 in (4, 6):
        shape["k"] = k2
        ids, w, _, _ = _screened_vs_fixed(shape, x.cuda(), w_r.cuda(), bias.cuda())
        ref_ids, ref_w, _ = oracle.route(bits(x), bits(w_r), bias.numpy(), G, tg, k2,
                                         SCORE_SIGMOID_BIAS)
        assert np.array_equal(ids, ref_ids)
        assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))


def _decode_router_inputs(T=512, seed=21):
    g = torch.Generator().manual_seed(seed)
    d, E = 7168, 256
    w_r = (torch.randn(d, E, generator=g) * 0.02)
    bias = torch.randn(E, generator=g, dtype=torch.float32)
    x = torch.randn(T, d, generator=g)
    return x, w_r, bias


@pytest.mark.parametrize("what", ["x*64", "x/64", "w_r*8", "outlier_columns", "x*64,w_r*8"])
def test_screened_route_large_and_outlier_inputs(what):
    # the regimes where tensor-core accumulation error is largest relative
    # to the score gaps: scaled activations and weights, and a few hidden
    # channels of magnitude ~100 in every token
    ensure_lib()
    from tests.gpu_common import bits
    cfg = CONFIGS["decode"]
    x, w_r, bias = _decode_router_inputs()
    base_shape = cfg.replace(T=x.shape[0]).shape()
    x0b, w0b = x.to(torch.bfloat16), w_r.to(torch.bfloat16)
    for part in what.split(","):
        if part == "x*64":
            x = x * 64
        elif part == "x/64":
            x = x / 64
        elif part == "w_r*8":
            w_r = w_r * 8
        elif part == "outlier_columns":
            cols = torch.tensor([7, 1000, 3333, 7000])
            x[:, cols] = 100.0 * torch.sign(x[:, cols])
    xb, wb = x.to(torch.bfloat16), w_r.to(torch.bfloat16)
    ids, w, _, n_ref = _screened_vs_fixed(base_shape, xb.cuda(), wb.cuda(), bias.cuda())
    ref_ids, ref_w, _ = oracle.route(bits(xb), bits(wb), bias.numpy(), cfg.G, cfg.topk_group,
                                     cfg.k, cfg.score)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))
    # the same tokens unscaled refine fewer pairs than the scaled ones
    _, _, _, n_ref0 = _screened_vs_fixed(base_shape, x0b.cuda(), w0b.cuda(), bias.cuda())
    print(f"{what}: refined pairs {n_ref} (unscaled {n_ref0}, T*k = {base_shape['T'] * cfg.k})")
    if what != "x/64":
        assert n_ref > n_ref0


def test_screened_route_engineered_near_ties():
    # groups come in twins: group 2q+1's weight columns are group 2q's with
    # one entry per column moved by one bf16 step, and twins share their
    # bias.  A twin pair's scores then differ by a few units in the last
    # place of the logit (far inside the tensor-core error bound).  With an
    # odd topk_group the group cut splits a twin pair, and with an odd k the
    # expert cut splits a pair of twin experts, in every token.
    ensure_lib()
    from tests.gpu_common import bits
    T, d, E, G, tg, k = 384, 2048, 128, 8, 3, 7
    gs = E // G
    g = torch.Generator().manual_seed(17)
    half = (torch.randn(d, E // 2, generator=g) * 0.03).to(torch.bfloat16)
    w_r = torch.empty(d, E, dtype=torch.bfloat16)
    for q in range(G):
        w_r[:, q * gs:(q + 1) * gs] = half[:, (q // 2) * gs:(q // 2 + 1) * gs]
    wbits = w_r.view(torch.int16)
    for q in range(1, G, 2):
        wbits[5, q * gs:(q + 1) * gs] += 1  # one bf16 step away from zero
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    hb = (torch.randn(E // 2, generator=g) * 0.01).to(torch.float32)
    bias = torch.empty(E, dtype=torch.float32)
    for q in range(G):
        bias[q * gs:(q + 1) * gs] = hb[(q // 2) * gs:(q // 2 + 1) * gs]
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    ids, w, _, n_ref = _screened_vs_fixed(shape, x.cuda(), w_r.cuda(), bias.cuda())
    ref_ids, ref_w, _ = oracle.route(bits(x), bits(w_r), bias.numpy(), G, tg, k,
                                     SCORE_SIGMOID_BIAS)
    assert np.array_equal(ids, ref_ids)
    assert np.all(np.abs(w - ref_w) <= 1e-6 * np.abs(ref_w))
    print(f"near ties: refined pairs {n_ref} ({n_ref / T:.1f} per token, k = {k})")
    assert n_ref >= T * (k + 1)


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_screened_route_full_size(name):
    ensure_lib()
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    ids, w, logits, n_ref = _screened_vs_fixed(cfg.shape(), t["x"], t["w_r"], t["bias"])
    # the fixed-order path itself is pinned to the oracle in
    # test_route_bit_exact_full_size; the intervals leave few experts open
    print(f"{name}: refined pairs {n_ref} = {n_ref / cfg.T:.2f} per token (k = {cfg.k})")
    assert n_ref < 2 * cfg.T * cfg.k


def test_prepared_router_weight_is_used_and_released():
    ensure_lib()
    import moe_inputs
    T, d, E = 300, 1024, 128
    shape = dict(T=T, d=d, E=E, G=4, topk_group=2, k=6, inter=64, score=SCORE_SIGMOID_BIAS,
                 bias_scale=0.15)
    a = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=41)
    b = moe_inputs.make_tensors_for_shape(T, d, E, 64, device="cuda", seed=42)
    ws = moe.Workspace(moe.moe_workspace_size(shape))

    def route(t):
        return [v.cpu() for v in moe.moe_route(shape, a["x"], t["w_r"], t["bias"], ws)[:2]]

    fresh = {"a": route(a), "b": route(b)}
    with moe.moe_router_prepare(shape, a["w_r"]) as prep:
        assert prep.buf.numel() >= moe.moe_router_prep_size(shape)
        for key, t in (("a", a), ("b", b), ("a", a)):
            got = route(t)
            assert torch.equal(got[0], fresh[key][0]) and torch.equal(got[1], fresh[key][1]), key
        # the record is used: a prepared copy of b's weight under a's pointer
        # (planted for the test) changes a's routing to b's
        n = moe.moe_router_prep_size(shape)

        def region(p):
            off = p.ptr - p.buf.data_ptr()
            return p.buf[off:off + n]

        with moe.moe_router_prepare(shape, b["w_r"]) as prep_b:
            saved = region(prep).clone()
            region(prep).copy_(region(prep_b))
            got = route(a)
            ref = [v.cpu() for v in moe.moe_route(shape, a["x"], b["w_r"], a["bias"], ws)[:2]]
            assert torch.equal(got[0], ref[0])
            region(prep).copy_(saved)
    # released: a's own weight again
    got = route(a)
    assert torch.equal(got[0], fresh["a"][0]) and torch.equal(got[1], fresh["a"][1])
    assert moe.moe_get_device_status(ws) == 0
    small = dict(shape, E=16, G=4)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_router_prepare(small, a["w_r"][:, :16].contiguous())
    assert ei.value.status == 2  # not screened


def test_refined_count_is_minus_one_when_not_screened():
    ensure_lib()
    import moe_inputs
    # E = 16 (not a multiple of 64): the fixed-order path
    tns = moe_inputs.make_tensors_for_shape(64, 256, 16, 64, device="cuda", seed=2)
    shape = dict(T=64, d=256, E=16, G=4, topk_group=2, k=2, inter=64,
                 score=SCORE_SIGMOID_BIAS, bias_scale=0.15)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    moe.moe_route(shape, tns["x"], tns["w_r"], tns["bias"], ws)
    assert moe.moe_route_refined_count(shape, ws) == -1
