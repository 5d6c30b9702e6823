"""The whole layer (moe_layer, the call bench.py times) and the masked
per-rank expert slices against the oracle, at the full workload sizes:
routing and counts bit-exact for every token, outputs of sampled tokens
(or rows) within the stated tolerance."""
import functools

import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import (CONFIGS, MASKED_EP_EXPERTS, MASKED_ROUTE_TOKENS, MASKED_TP_INTER,
                        SCORE_SIGMOID_BIAS, make_layer_tensors)
from tests.gpu_common import bits, check_close, ensure_lib, host_bits, layer_inputs

pytestmark = pytest.mark.gpu

SAMPLES = {"tiny": None, "few_large": 16, "decode": 16, "prefill": 8}


@functools.lru_cache(maxsize=None)
def oracle_routing(name):
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    logits = oracle.router_logits(host_bits(name, "x"), host_bits(name, "w_r"))
    ids, w, _ = oracle.route_from_logits(logits, t["bias"].cpu().numpy(), cfg.G,
                                         cfg.topk_group, cfg.k, cfg.score, cfg.bias_scale)
    return ids, w


@pytest.mark.parametrize("name", ["tiny", "few_large", "decode", "prefill"])
def test_layer_matches_oracle(name):
    ensure_lib()
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    bias = t["bias"] if cfg.score == SCORE_SIGMOID_BIAS else None
    y = moe.moe_layer(cfg.shape(), t["x"], t["w_r"], bias, t["w_gate_up"], t["w_down"], ws,
                      topk_ids=ids, topk_w=w, counts=counts)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ref_ids, ref_w = oracle_routing(name)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    gw = w.cpu().numpy()
    assert np.all(np.abs(gw - ref_w) <= 1e-6 * np.abs(ref_w))
    assert np.array_equal(counts.cpu().numpy(), np.bincount(ref_ids.ravel(), minlength=cfg.E))
    # outputs of sampled tokens (all tokens for the tiny workload)
    n = SAMPLES[name]
    if n is None:
        toks = np.arange(cfg.T, dtype=np.int32)
    else:
        rng = np.random.default_rng(0)
        toks = np.sort(rng.choice(cfg.T, n, replace=False)).astype(np.int32)
        toks[0] = 0
        toks[-1] = cfg.T - 1
    y_ref, ids_t, _ = oracle.layer_tokens(host_bits(name, "x"), host_bits(name, "w_r"),
                                          t["bias"].cpu().numpy(), host_bits(name, "w_gate_up"),
                                          host_bits(name, "w_down"), cfg.shape(), toks)
    assert np.array_equal(ids_t, ref_ids[toks])
    got = y.float().cpu().numpy()[toks]
    check_close(got, y_ref, bf16_output=True, what=name)


def test_layer_is_deterministic_and_repeatable():
    ensure_lib()
    cfg = CONFIGS["tiny"]
    t = layer_inputs("tiny")
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    ys = [moe.moe_layer(cfg.shape(), t["x"], t["w_r"], t["bias"], t["w_gate_up"],
                        t["w_down"], ws) for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_layer_single_token_and_ragged_T():
    ensure_lib()
    base = CONFIGS["tiny"]
    t = layer_inputs("tiny")
    for T in (1, 3, 37):
        cfg = base.replace(T=T)
        x = t["x"][:T].contiguous()
        ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
        y = moe.moe_layer(cfg.shape(), x, t["w_r"], t["bias"], t["w_gate_up"], t["w_down"], ws)
        y_ref, _, _ = oracle.layer_tokens(bits(x), host_bits("tiny", "w_r"),
                                          t["bias"].cpu().numpy(),
                                          host_bits("tiny", "w_gate_up"),
                                          host_bits("tiny", "w_down"), cfg.shape(),
                                          np.arange(T, dtype=np.int32))
        check_close(y.float().cpu().numpy(), y_ref, bf16_output=True, what=f"T={T}")


# ---------------------------------------------------------------------------
# masked per-rank expert slices
# ---------------------------------------------------------------------------

@functools.lru_cache(maxsize=None)
def masked_source():
    """4096 tokens routed through the decode router (oracle routing)."""
    cfg = CONFIGS["decode"]
    t = make_layer_tensors(cfg, device="cuda", seed=0, n_tokens=MASKED_ROUTE_TOKENS)
    xb = bits(t["x"])
    logits = oracle.router_logits(xb, bits(t["w_r"]))
    ids, _, _ = oracle.route_from_logits(logits, t["bias"].cpu().numpy(), cfg.G,
                                         cfg.topk_group, cfg.k, cfg.score, cfg.bias_scale)
    counts, offsets, dest, src = oracle.dispatch(ids, cfg.E)
    return t, xb, counts, offsets, src


def _masked_buffer(x, src, offsets, experts, M_max):
    E_l = len(experts)
    buf = torch.zeros(E_l, M_max, x.shape[1], dtype=torch.bfloat16, device="cuda")
    mm = []
    for i, e in enumerate(experts):
        rows = torch.from_numpy(src[offsets[e]:offsets[e + 1]].astype(np.int64)).cuda()
        buf[i, :rows.numel()] = x[rows]
        mm.append(rows.numel())
    return buf, torch.tensor(mm, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("variant", ["ep", "tp"])
def test_masked_expert_slices(variant):
    ensure_lib()
    cfg = CONFIGS["decode"]
    t, xb, counts, offsets, src = masked_source()
    if variant == "ep":
        experts = list(range(MASKED_EP_EXPERTS))
        w_gu = t["w_gate_up"][:MASKED_EP_EXPERTS].contiguous()
        w_down = t["w_down"][:MASKED_EP_EXPERTS].contiguous()
        inter = cfg.inter
    else:
        experts = list(range(cfg.E))
        i0 = MASKED_TP_INTER
        w_gu = torch.cat([t["w_gate_up"][:, :i0], t["w_gate_up"][:, cfg.inter:cfg.inter + i0]],
                         dim=1).contiguous()
        w_down = t["w_down"][:, :, :i0].contiguous()
        inter = i0
    mm_host = counts[experts]
    M_max = max(128, int(-(-mm_host.max() // 128) * 128))
    buf, mm = _masked_buffer(t["x"], src, offsets, experts, M_max)
    shape = dict(T=1, d=cfg.d, E=len(experts), G=1, topk_group=1, k=1, inter=inter, score=1,
                 bias_scale=0.15)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_MASKED, M_max))
    y = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_MASKED, buf, mm, M_max, w_gu, w_down, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    # sampled rows: first/last row of the busiest experts and of a few others
    order = np.argsort(-mm_host, kind="stable")
    pick_e = [int(e) for e in order[:4]] + [int(e) for e in order[4:] if mm_host[e] > 0][:4]
    rows, row_e = [], []
    for i in pick_e:
        m = int(mm_host[i])
        for r in sorted({0, m // 2, m - 1}):
            rows.append((i, r))
            row_e.append(i)
    xr = np.stack([bits(buf[i, r]) for i, r in rows])
    ref = oracle.expert_ffn_rows(xr, np.array(row_e, np.int32), bits(w_gu), bits(w_down))
    got = np.stack([y[i, r].cpu().numpy() for i, r in rows])
    check_close(got, ref, bf16_output=False, what=f"masked {variant}")
