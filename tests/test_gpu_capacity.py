"""Capacity variant ("第十五章" section 4.3, "Capacity Factor" and the
overflow table) against the oracle: the capacity dispatch bit-exact, the
layer with dropped or second-round overflow within the stated tolerance,
and the second round equal to the uncapped layer."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import CONFIGS, SCORE_SIGMOID_BIAS, random_ids
from tests.gpu_common import bf16_to_f64, bits, check_close, ensure_lib, host_bits, layer_inputs
from tests.test_gpu_layer import oracle_routing

pytestmark = pytest.mark.gpu


def _shape(T, d, E, k):
    return dict(T=T, d=d, E=E, G=1, topk_group=1, k=k, inter=64, score=1, bias_scale=0.15)


@pytest.mark.parametrize("T,k,E,d,C,skew", [
    (1000, 8, 256, 64, 40, 2.0),     # decode-like: hot experts overflow
    (513, 4, 5, 24, 300, 0.0),       # nothing overflows
    (300, 2, 7, 16, 0, 1.0),         # capacity 0: everything overflows
    (4096, 2, 8, 128, 460, 0.3),     # few_large-like with c ~ 0.9
    (37, 3, 3, 8, 5, 3.0),
])
@pytest.mark.parametrize("policy", [moe.MOE_OVERFLOW_DROP, moe.MOE_OVERFLOW_SECOND_ROUND])
def test_dispatch_capacity_bit_exact(T, k, E, d, C, skew, policy):
    ensure_lib()
    ids = random_ids(T, k, E, seed=T + C, skew=skew)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    shape = _shape(T, d, E, k)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    counts, kept, ovf, dest, src, x_rows = moe.moe_dispatch_capacity(shape, C, policy,
                                                                     ids.cuda(), x.cuda(), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    r_counts, r_kept, r_ovf, r_dest, r_src = oracle.dispatch_capacity(ids.numpy(), E, C, policy)
    assert np.array_equal(counts.cpu().numpy(), r_counts)
    assert np.array_equal(kept.cpu().numpy(), r_kept)
    assert np.array_equal(ovf.cpu().numpy(), r_ovf)
    assert np.array_equal(dest.cpu().numpy(), r_dest)
    used = r_src >= 0
    assert np.array_equal(src.cpu().numpy()[used], r_src[used])
    xb = bits(x)
    assert np.array_equal(bits(x_rows.cpu())[used], xb[r_src[used]])


def _capacity_layer(name, C, policy):
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    shape = cfg.shape()
    ws = moe.Workspace(moe.moe_layer_capacity_workspace_size(shape, C))
    bias = t["bias"] if cfg.score == SCORE_SIGMOID_BIAS else None
    kept = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    y = moe.moe_layer_capacity(shape, C, policy, t["x"], t["w_r"], bias, t["w_gate_up"],
                               t["w_down"], ws, kept=kept)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return y, kept.cpu().numpy()


@pytest.mark.parametrize("name,c,n_samples", [
    ("tiny", 1.0, None), ("tiny", 0.5, None), ("decode", 1.0, 24), ("few_large", 0.95, 12)])
@pytest.mark.parametrize("policy", [moe.MOE_OVERFLOW_DROP, moe.MOE_OVERFLOW_SECOND_ROUND])
def test_layer_capacity_matches_oracle(name, c, n_samples, policy):
    ensure_lib()
    cfg = CONFIGS[name]
    C = moe.moe_expert_capacity(cfg.T, cfg.k, cfg.E, c)
    assert C == oracle.expert_capacity(cfg.T, cfg.k, cfg.E, c)
    y, kept = _capacity_layer(name, C, policy)
    ids, _ = oracle_routing(name)
    counts, r_kept, _, dest, _ = oracle.dispatch_capacity(ids, cfg.E, C, policy)
    assert np.array_equal(kept, r_kept)
    if policy == moe.MOE_OVERFLOW_DROP:
        assert (counts > C).any(), "the case must overflow"
    if n_samples is None:
        toks = np.arange(cfg.T, dtype=np.int32)
    else:
        rng = np.random.default_rng(1)
        toks = np.sort(rng.choice(cfg.T, n_samples, replace=False)).astype(np.int32)
        # include tokens that lost an assignment
        lost = np.where((dest.reshape(cfg.T, cfg.k) < 0).any(1))[0]
        if lost.size:
            toks = np.unique(np.concatenate([toks, lost[:4]])).astype(np.int32)
    keep = (dest.reshape(cfg.T, cfg.k)[toks] >= 0).astype(np.uint8)
    t = layer_inputs(name)
    y_ref, _, _ = oracle.layer_tokens(host_bits(name, "x"), host_bits(name, "w_r"),
                                      t["bias"].cpu().numpy(), host_bits(name, "w_gate_up"),
                                      host_bits(name, "w_down"), cfg.shape(), toks, keep=keep)
    got = bf16_to_f64(y[torch.from_numpy(toks).cuda().long()])
    check_close(got, y_ref, bf16_output=True, what=f"{name} capacity {C} policy {policy}")


def test_capacity_zero_drop_gives_zero_and_second_round_gives_full_layer():
    ensure_lib()
    cfg = CONFIGS["tiny"]
    y0, kept = _capacity_layer("tiny", 0, moe.MOE_OVERFLOW_DROP)
    assert not kept.any()
    assert not y0.float().abs().max().item()
    y2, _ = _capacity_layer("tiny", 0, moe.MOE_OVERFLOW_SECOND_ROUND)
    t = layer_inputs("tiny")
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    y = moe.moe_layer(cfg.shape(), t["x"], t["w_r"], t["bias"], t["w_gate_up"], t["w_down"], ws)
    torch.cuda.synchronize()
    # same rows, same kernels, same per-row arithmetic
    assert torch.equal(y2, y)
