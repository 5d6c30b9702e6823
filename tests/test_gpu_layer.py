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

# tokens whose outputs are compared: every token of the small workloads;
# at few_large and prefill a set that covers the first and the last row of
# every 128-row m-tile of every touched expert
ALL_TOKENS = {"tiny", "decode"}
TILE = 128


def tile_cover_tokens(ids: np.ndarray, E: int):
    """Tokens whose assignments include the first and the last row of every
    128-row m-tile of every expert, from the oracle's dispatch of the oracle
    routing.  Returns (tokens, number of m-tiles)."""
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    rows = []
    n_tiles = 0
    for e in range(E):
        n = int(counts[e])
        for j in range(0, n, TILE):
            n_tiles += 1
            rows += [int(offsets[e]) + j, int(offsets[e]) + min(j + TILE, n) - 1]
    return np.unique(src[np.array(rows, dtype=np.int64)]).astype(np.int32), n_tiles


def tiles_covered(ids: np.ndarray, E: int, toks: np.ndarray) -> int:
    """m-tiles whose first and last rows both belong to assignments of `toks`."""
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    k = ids.shape[1]
    have = np.zeros(ids.size, dtype=bool)
    have[dest[(toks[:, None].astype(np.int64) * k + np.arange(k)).ravel()]] = True
    covered = 0
    for e in range(E):
        n = int(counts[e])
        for j in range(0, n, TILE):
            covered += int(have[offsets[e] + j] and have[offsets[e] + min(j + TILE, n) - 1])
    return covered


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
    if name in ALL_TOKENS:
        toks = np.arange(cfg.T, dtype=np.int32)
        _, n_tiles = tile_cover_tokens(ref_ids, cfg.E)
    else:
        toks, n_tiles = tile_cover_tokens(ref_ids, cfg.E)
    covered = tiles_covered(ref_ids, cfg.E, toks)
    print(f"{name}: {len(toks)} of {cfg.T} tokens compared, m-tiles covered "
          f"{covered} of {n_tiles}")
    assert covered == n_tiles
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


def test_layer_fp32_rows_where_d_is_not_a_multiple_of_256():
    """d = 448: the layer keeps the down GEMM's rows in fp32 (the compact form
    needs whole 256-column tiles) and combines them with the fp32 combine;
    every token against the oracle."""
    ensure_lib()
    import moe_inputs
    T, d, E, inter = 96, 448, 8, 128
    cfg = CONFIGS["tiny"].replace(T=T, d=d, E=E, G=2, topk_group=1, k=2, inter=inter,
                                  name="d448")
    shape = cfg.shape()
    assert moe.moe_layer_yperm_row_bytes(shape) == 4 * d
    t = moe_inputs.make_layer_tensors(cfg, device="cuda", seed=448)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    y = moe.moe_layer(shape, t["x"], t["w_r"], t["bias"], t["w_gate_up"], t["w_down"], ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    y_ref, _, _ = oracle.layer_tokens(bits(t["x"]), bits(t["w_r"]), t["bias"].cpu().numpy(),
                                      bits(t["w_gate_up"]), bits(t["w_down"]), shape,
                                      np.arange(T, dtype=np.int32))
    check_close(y.float().cpu().numpy(), y_ref, bf16_output=True, what="d=448")


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
    # the first and the last row of every 128-row m-tile of every slab
    rows, row_e = [], []
    n_tiles = 0
    for i in range(len(experts)):
        m = int(mm_host[i])
        for j in range(0, m, TILE):
            n_tiles += 1
            for r in sorted({j, min(j + TILE, m) - 1}):
                rows.append((i, r))
                row_e.append(i)
    have = set(rows)
    covered = sum(1 for i in range(len(experts)) for j in range(0, int(mm_host[i]), TILE)
                  if (i, j) in have and (i, min(j + TILE, int(mm_host[i])) - 1) in have)
    print(f"masked {variant}: {len(rows)} rows compared, m-tiles covered {covered} of {n_tiles}")
    assert covered == n_tiles
    idx_i = torch.tensor([i for i, _ in rows], device="cuda")
    idx_r = torch.tensor([r for _, r in rows], device="cuda")
    xr = bits(buf[idx_i, idx_r])
    ref = oracle.expert_ffn_rows(xr, np.array(row_e, np.int32), bits(w_gu), bits(w_down))
    got = y[idx_i, idx_r].cpu().numpy()
    check_close(got, ref, bf16_output=False, what=f"masked {variant}")


@pytest.mark.parametrize("name", ["tiny", "few_large", "decode", "prefill"])
def test_layer_compact_rows_within_their_bound(name):
    """With d a multiple of 256 the layer keeps the down GEMM's rows (1-CTA
    or CTA-pair form) as fp16 values with a power-of-two scale per 32 columns.
    Against the same layer composed from the public calls (fp32 rows), every
    output differs by at most that form's rounding -- 2^-11 of each group's
    largest magnitude, weighted like the combine -- plus one bf16 step."""
    ensure_lib()
    cfg = CONFIGS[name]
    shape = cfg.shape()
    d = cfg.d
    assert moe.moe_layer_yperm_row_bytes(shape) == 2 * d + d // 32
    t = layer_inputs(name)
    bias = t["bias"] if cfg.score == SCORE_SIGMOID_BIAS else None
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    y = moe.moe_layer(shape, t["x"], t["w_r"], bias, t["w_gate_up"], t["w_down"], ws)
    ids, w, _ = moe.moe_route(shape, t["x"], t["w_r"], bias, ws)
    _, offsets, _, dest, x_perm = moe.moe_dispatch(shape, ids, t["x"], ws)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y_perm = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x_perm, offsets, 0,
                                t["w_gate_up"], t["w_down"], fws)
    y_ref = moe.moe_combine(shape, y_perm, dest, w)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0 and moe.moe_get_device_status(fws) == 0
    del x_perm, fws
    T, k = cfg.T, cfg.k
    gmax = y_perm.abs().view(-1, d // 32, 32).amax(-1)               # [T*k, d/32]
    rows = dest.view(T, k).long()
    bound = (w.abs().unsqueeze(-1) * gmax[rows]).sum(1) * 2.0 ** -11  # [T, d/32]
    bound = bound.repeat_interleave(32, dim=1)
    yr = y_ref.float()
    mag = yr.abs() + bound
    ulp = torch.where(mag > 0, torch.exp2(torch.floor(torch.log2(mag)) - 7),
                      torch.zeros_like(mag))
    excess = ((y.float() - yr).abs() - bound - ulp).max().item()
    assert excess <= 0.0, f"{name}: compact rows exceed their bound by {excess:.3e}"
    same = (y.view(torch.int16) == y_ref.view(torch.int16)).float().mean().item()
    print(f"{name}: {same * 100:.2f} % of outputs identical to the fp32-row composition")


@pytest.mark.parametrize("scale_exp", [40, -60, -118])
def test_layer_compact_rows_extreme_magnitudes(scale_exp):
    """The compact rows keep their bound for outputs of any magnitude: the
    tiny layer with its down weights scaled by 2^scale_exp (outputs near
    2^40, 2^-60, and below the form's floor of 2^-111, where a group is
    stored as zero) against the fp32-row composition of the public calls."""
    ensure_lib()
    cfg = CONFIGS["tiny"]
    shape = cfg.shape()
    d = cfg.d
    t = layer_inputs("tiny")
    w_down = (t["w_down"].float() * 2.0 ** scale_exp).to(torch.bfloat16)
    bias = t["bias"] if cfg.score == SCORE_SIGMOID_BIAS else None
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    y = moe.moe_layer(shape, t["x"], t["w_r"], bias, t["w_gate_up"], w_down, ws)
    ids, w, _ = moe.moe_route(shape, t["x"], t["w_r"], bias, ws)
    _, offsets, _, dest, x_perm = moe.moe_dispatch(shape, ids, t["x"], ws)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y_perm = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x_perm, offsets, 0,
                                t["w_gate_up"], w_down, fws)
    y_ref = moe.moe_combine(shape, y_perm, dest, w)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    T, k = cfg.T, cfg.k
    gmax = y_perm.abs().view(-1, d // 32, 32).amax(-1)
    # rounding 2^-11 of the group's largest value; below 2^-111 the group is zero
    gerr = torch.where(gmax >= 2.0 ** -111, gmax * 2.0 ** -11, gmax)
    bound = (w.abs().unsqueeze(-1) * gerr[dest.view(T, k).long()]).sum(1)
    bound = bound.repeat_interleave(32, dim=1)
    yr = y_ref.float()
    mag = yr.abs() + bound
    ulp = torch.where(mag > 0, torch.exp2(torch.floor(torch.log2(mag)) - 7),
                      torch.zeros_like(mag))
    # the bf16 step of the smallest normal where the magnitudes are subnormal
    ulp = torch.maximum(ulp, torch.full_like(ulp, 2.0 ** -133))
    assert torch.isfinite(y.float()).all()
    excess = ((y.float() - yr).abs() - bound - ulp).max().item()
    assert excess <= 0.0, f"scale 2^{scale_exp}: excess {excess:.3e}"
    if scale_exp < -111:  # most groups under the floor: stored, and summed, as zero
        assert float(yr.abs().max()) > 0.0
        assert float((y.float() == 0).float().mean()) > 0.5
