"""Dispatch onto physical expert copies (moe_dispatch_replicated) against the
oracle, bit for bit, and an MoE layer run on the physical layout with
replicated weights against the oracle layer.  Pages: "ep-deploy" handbook,
section "EPLB 与路由约束" (copies of hot experts, their placement), and
"第十五章" section 4.3 (each assignment goes to one of its expert's
equivalent copies)."""
import ctypes

import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import CONFIGS, SCORE_SIGMOID_BIAS, make_tensors_for_shape, random_ids
from tests.gpu_common import bits, check_close, ensure_lib

pytestmark = pytest.mark.gpu


def _shape(T, d, E, k):
    return dict(T=T, d=d, E=E, G=1, topk_group=1, k=k, inter=64, score=1, bias_scale=0.15)


def _run(ids, x, E, phys):
    T, k = ids.shape
    shape = _shape(T, x.shape[1] if x is not None else 64, E, k)
    ws = moe.Workspace(moe.moe_dispatch_replicated_workspace_size(shape, len(phys)))
    pe = torch.from_numpy(np.asarray(phys, np.int32)).cuda()
    out = moe.moe_dispatch_replicated(shape, pe, ids.cuda(), x, ws)
    torch.cuda.synchronize()
    return out, ws


def _check(ids, x, E, phys):
    (counts, offsets, src, dest, xp), ws = _run(ids, x, E, phys)
    assert moe.moe_get_device_status(ws) == 0
    rc, ro, rd, rs = oracle.dispatch_replicated(ids.numpy(), E, np.asarray(phys, np.int32))
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(dest.cpu().numpy(), rd)
    assert np.array_equal(src.cpu().numpy(), rs)
    if x is not None:
        assert np.array_equal(bits(xp), bits(x)[rs])


@pytest.mark.parametrize("T,k,E,P,d,skew,seed", [
    (257, 4, 16, 16, 64, 0.0, 0),      # one copy each, shuffled slots
    (1000, 8, 64, 96, 128, 2.0, 1),    # hot experts with extra copies
    (33, 2, 8, 40, 256, 1.0, 2),       # five copies per expert on average, few rows
    (4096, 8, 256, 288, 64, 2.5, 3),   # the page's 32-GPU prefill shape: 9 slots per GPU
    (5000, 8, 256, 1100, 16, 1.5, 4),  # more slots than one 1024-thread pass
    (70000, 2, 32, 64, 16, 1.0, 5),    # T*k > 32768: 512-assignment chunks
])
def test_replicated_dispatch_bit_exact(T, k, E, P, d, skew, seed):
    ensure_lib()
    rng = np.random.default_rng(seed)
    ids = random_ids(T, k, E, seed=seed, skew=skew)
    n_e = np.bincount(ids.numpy().ravel(), minlength=E)
    extra = rng.choice(E, P - E, p=(n_e + 1) / (n_e + 1).sum()) if P > E else []
    phys = np.concatenate([np.arange(E), extra]).astype(np.int32)
    rng.shuffle(phys)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).cuda()
    _check(ids, x, E, phys)


def test_identity_placement_is_moe_dispatch():
    ensure_lib()
    T, k, E, d = 999, 6, 48, 128
    ids = random_ids(T, k, E, seed=8, skew=1.5)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16).cuda()
    (counts, offsets, src, dest, xp), _ = _run(ids, x, E, np.arange(E))
    shape = _shape(T, d, E, k)
    ref = moe.moe_dispatch(shape, ids.cuda(), x, moe.Workspace(moe.moe_workspace_size(shape)))
    for g, r in zip((counts, offsets, src, dest), ref[:4]):
        assert torch.equal(g, r)
    assert np.array_equal(bits(xp), bits(ref[4]))


def test_planner_placement_on_decode_routing():
    # the decode router's assignment counts -> the planner's global placement
    # on 32 GPUs with 32 extra copies -> the dispatch of those assignments
    ensure_lib()
    from tests.test_gpu_layer import oracle_routing
    cfg = CONFIGS["decode"]
    ids, _ = oracle_routing("decode")
    load = np.bincount(ids.ravel(), minlength=cfg.E).astype(np.float64)
    slots, reps = moe.moe_eplb_plan(load, cfg.G, 0, 32, cfg.E + 32)
    phys = np.asarray(slots, np.int32).reshape(-1)
    _check(torch.from_numpy(ids), None, cfg.E, phys)
    (counts, offsets, _, _, _), _ = _run(torch.from_numpy(ids), None, cfg.E, phys)
    per_gpu = counts.cpu().numpy().reshape(32, -1).sum(1)
    # copies spread the hot experts over the GPUs (the placement's purpose)
    assert per_gpu.max() / per_gpu.mean() < 1.5


def test_routed_expert_without_copy_is_flagged():
    ensure_lib()
    ids = torch.tensor([[0, 1], [2, 1]], dtype=torch.int32)
    (counts, offsets, src, dest, _), ws = _run(ids, None, 4, np.array([0, 2, 3, 0], np.int32))
    assert moe.moe_get_device_status(ws) == 1  # MOE_ERR_INVALID_ARG
    d = dest.cpu().numpy()
    assert d[1] == -1 and d[3] == -1
    assert np.array_equal(counts.cpu().numpy(), [1, 1, 0, 0])


def test_layer_on_replicated_experts_matches_oracle():
    # route, place copies of the hot experts, dispatch onto the copies, run
    # the expert FFN over the physical slots with replicated weights, combine:
    # the output is the layer's, whichever copy a token met
    ensure_lib()
    T, d, E, inter, G, tg, k = 512, 1024, 32, 256, 4, 2, 4
    t = make_tensors_for_shape(T, d, E, inter, device="cuda", seed=23, w_std=0.03)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=inter,
                 score=SCORE_SIGMOID_BIAS, bias_scale=0.15)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    ids, w, _ = moe.moe_route(shape, t["x"], t["w_r"], t["bias"], ws)
    load = np.bincount(ids.cpu().numpy().ravel(), minlength=E).astype(np.float64)
    slots, _ = moe.moe_eplb_plan(load, G, 0, 8, E + 16)
    phys = torch.from_numpy(np.asarray(slots, np.int32).reshape(-1)).cuda()
    P = phys.numel()
    rws = moe.Workspace(moe.moe_dispatch_replicated_workspace_size(shape, P))
    counts, offsets, src, dest, xp = moe.moe_dispatch_replicated(shape, phys, ids, t["x"], rws)
    fshape = dict(T=T * k, d=d, E=P, G=1, topk_group=1, k=1, inter=inter, score=1,
                  bias_scale=0.15)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(fshape, moe.MOE_LAYOUT_CONTIGUOUS))
    w_gu = t["w_gate_up"][phys.long()].contiguous()
    w_dn = t["w_down"][phys.long()].contiguous()
    y_perm = moe.moe_expert_ffn(fshape, moe.MOE_LAYOUT_CONTIGUOUS, xp, offsets, 0, w_gu, w_dn,
                                fws)
    y = moe.moe_combine(shape, y_perm, dest, w)
    y_layer = moe.moe_layer(shape, t["x"], t["w_r"], t["bias"], t["w_gate_up"], t["w_down"], ws)
    torch.cuda.synchronize()
    for wsx in (ws, rws, fws):
        assert moe.moe_get_device_status(wsx) == 0
    assert int(counts.sum()) == T * k and (counts > 0).sum() > E  # copies in use
    y_ref, _, _ = oracle.layer_tokens(bits(t["x"]), bits(t["w_r"]), t["bias"].cpu().numpy(),
                                      bits(t["w_gate_up"]), bits(t["w_down"]), shape,
                                      np.arange(T, dtype=np.int32))
    check_close(y.float().cpu().numpy(), y_ref, bf16_output=True, what="replicated layer")
    check_close(y_layer.float().cpu().numpy(), y_ref, bf16_output=True, what="layer")
