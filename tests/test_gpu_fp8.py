"""FP8 path (e4m3 codes with power-of-two fp32 block scales) against the oracle: the
quantizers bit-exact, the FP8 expert FFN (contiguous and masked layouts,
ragged tiles) and the FP8 layer within the stated tolerance."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import CONFIGS, SCORE_SIGMOID_BIAS
from tests.gpu_common import bf16_to_f64, bits, check_close, ensure_lib, host_bits, layer_inputs
from tests.test_gpu_layer import oracle_routing, tile_cover_tokens, tiles_covered

pytestmark = pytest.mark.gpu


def _rand_bf16(shape, seed, scale_cols=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    if scale_cols is not None:
        x = x * scale_cols
    return x.to(torch.bfloat16)


def test_quantize_rows_bit_exact():
    ensure_lib()
    mags = torch.tensor([1e-4, 1.0, 300.0, 1e3]).repeat_interleave(128)
    x = _rand_bf16((333, 512), 1, mags)
    x[7, 128:256] = 0                       # all-zero block: scale 1
    x[9, 0] = 448.0                         # exact code boundaries
    q, s = moe.moe_quantize_fp8_rows(x.cuda())
    rq, rs = oracle.quantize_rows_fp8(bits(x))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


def test_quantize_rows_scale_boundaries_bit_exact():
    # the power-of-two scale at its boundaries: amax exactly 448 * 2^k, the
    # next bf16 above it, values whose amax clamps the exponent at -127 (bf16
    # subnormals among them), amax near the bf16 maximum, an all-zero block;
    # each row one 128-column block, the rest of the row random
    ensure_lib()
    amaxes = [448.0, 448.0 * 2.0 ** -20, 448.0 * 2.0 ** 30, 450.0, 1.0, 1.75, 1.7578125,
              2.0 ** -130, 1e-38, 3.0e38, 0.0]
    x = _rand_bf16((len(amaxes), 256), 3) * 1e-3
    for r, a in enumerate(amaxes):
        x[r, :128] = 0.0
        x[r, 5] = a
        x[r, 9] = -0.75 * a
        x[r, 17] = a * 2.0 ** -12
    q, s = moe.moe_quantize_fp8_rows(x.cuda())
    rq, rs = oracle.quantize_rows_fp8(bits(x))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert rs[0, 0] == 1.0 and rs[3, 0] == 2.0 and rs[len(amaxes) - 1, 0] == 1.0


def test_quantize_blocks_bit_exact():
    ensure_lib()
    w = _rand_bf16((3, 256, 384), 2) * 0.02
    w[1, :128, 128:256] = 0
    q, s = moe.moe_quantize_fp8_blocks(w.cuda())
    rq, rs = oracle.quantize_blocks_fp8(bits(w))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


def _weights_fp8(E, d, inter, seed):
    w_gu = _rand_bf16((E, 2 * inter, d), seed) / d ** 0.5
    w_dn = _rand_bf16((E, d, inter), seed + 1) / inter ** 0.5
    gq, gs = moe.moe_quantize_fp8_blocks(w_gu.cuda())
    dq, ds = moe.moe_quantize_fp8_blocks(w_dn.cuda())
    rgq, rgs = oracle.quantize_blocks_fp8(bits(w_gu))
    rdq, rds = oracle.quantize_blocks_fp8(bits(w_dn))
    assert np.array_equal(gq.cpu().numpy(), rgq) and np.array_equal(dq.cpu().numpy(), rdq)
    return (gq, gs, dq, ds), (rgq, rgs, rdq, rds)


def _shape(E, d, inter, T):
    return dict(T=T, d=d, E=E, G=1, topk_group=1, k=1, inter=inter, score=1, bias_scale=0.15)


@pytest.mark.parametrize("counts,d,inter", [
    ([0, 1, 127, 128, 129, 300], 256, 128),
    ([5, 0, 260], 512, 256),
    ([40, 300, 1], 384, 384),
    ([3, 200], 4096, 1024),                 # long K in both GEMMs
    # >= 256 rows per expert: CTA-pair tiles of 256 rows (an expert of 5 rows
    # and tails of 1 and 255 rows leave the odd CTA of the pair empty or short)
    ([300, 700, 5, 600], 512, 256),
    ([256, 257, 511, 512, 1], 256, 128),
    ([1000, 1100], 1024, 512),
])
def test_ffn_fp8_contiguous(counts, d, inter):
    ensure_lib()
    E = len(counts)
    rows = sum(counts)
    x = _rand_bf16((rows, d), d + inter)
    (gq, gs, dq, ds), (rgq, rgs, rdq, rds) = _weights_fp8(E, d, inter, seed=d)
    xq, xs = moe.moe_quantize_fp8_rows(x.cuda())
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    shape = _shape(E, d, inter, rows)
    ws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_CONTIGUOUS, xq, xs, offsets, 0, gq, gs, dq,
                               ds, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    rxq, rxs = oracle.quantize_rows_fp8(bits(x))
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    ref = oracle.expert_ffn_rows_fp8(rxq, rxs, row_e, rgq, rgs, rdq, rds)
    check_close(y.cpu().numpy(), ref, bf16_output=False, what="y (fp8)")


def test_ffn_fp8_prefill_shape_every_tile():
    # the CTA-pair FP8 GEMMs (h quantized in the gate_up epilogue) at the
    # prefill expert shape, d = 7168 and inter = 2048, on a skewed mix of
    # expert row counts (an odd half with no rows, tails just under and over a
    # 128-row half, full and partial tiles): the first and the last row of
    # every 128-row m-tile compared with the oracle
    ensure_lib()
    counts = [5, 130, 255, 257, 601, 2413]
    E, d, inter = len(counts), 7168, 2048
    rows = sum(counts)
    x = _rand_bf16((rows, d), 21)
    (gq, gs, dq, ds), (rgq, rgs, rdq, rds) = _weights_fp8(E, d, inter, seed=22)
    xq, xs = moe.moe_quantize_fp8_rows(x.cuda())
    offs = np.concatenate([[0], np.cumsum(counts)])
    offsets = torch.tensor(offs, dtype=torch.int32).cuda()
    shape = _shape(E, d, inter, rows)   # rows / expert >= 256: CTA-pair tiles
    ws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_CONTIGUOUS, xq, xs, offsets, 0, gq, gs, dq,
                               ds, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    sel = sorted({int(offs[e]) + j for e, c in enumerate(counts) for t0 in range(0, c, 128)
                  for j in (t0, min(t0 + 128, c) - 1)})
    sel = np.array(sel, dtype=np.int64)
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)[sel]
    rxq, rxs = oracle.quantize_rows_fp8(bits(x)[sel])
    ref = oracle.expert_ffn_rows_fp8(rxq, rxs, row_e, rgq, rgs, rdq, rds)
    check_close(y.cpu().numpy()[sel], ref, bf16_output=False, what="y (fp8, prefill shape)")


@pytest.mark.parametrize("masked_m,M_max,T", [
    ([0, 5, 256], 256, 1),
    ([0, 5, 300, 512], 512, 1300),   # T*k >= 256 per expert and M_max >= 256: pair tiles
])
def test_ffn_fp8_masked(masked_m, M_max, T):
    ensure_lib()
    E, d, inter = len(masked_m), 256, 256
    x = _rand_bf16((E, M_max, d), 11)
    (gq, gs, dq, ds), (rgq, rgs, rdq, rds) = _weights_fp8(E, d, inter, seed=12)
    xq, xs = moe.moe_quantize_fp8_rows(x.reshape(E * M_max, d).cuda())
    shape = _shape(E, d, inter, T)
    ws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(shape, moe.MOE_LAYOUT_MASKED, M_max))
    mm = torch.tensor(masked_m, dtype=torch.int32).cuda()
    y = torch.full((E * M_max, d), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_MASKED, xq, xs, mm, M_max, gq, gs, dq, ds, ws,
                           y_out=y)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    rxq, rxs = oracle.quantize_rows_fp8(bits(x.reshape(E * M_max, d)))
    yc = y.cpu().numpy()
    for e, m in enumerate(masked_m):
        if m == 0:
            assert np.isnan(yc[e * M_max:(e + 1) * M_max]).all()
            continue
        rows = slice(e * M_max, e * M_max + m)
        ref = oracle.expert_ffn_rows_fp8(rxq[rows], rxs[rows], np.full(m, e, np.int32), rgq, rgs,
                                         rdq, rds)
        check_close(yc[rows], ref, bf16_output=False, what=f"expert {e}")
        assert np.isnan(yc[e * M_max + m:(e + 1) * M_max]).all()


@pytest.mark.parametrize("pair_rows", [False, True])
def test_ffn_fp8_flags_a_scale_that_is_not_a_power_of_two(pair_rows):
    # the tensor cores take each scale as an 8-bit exponent: any other value
    # is reported in the device status (1-CTA and CTA-pair forms)
    ensure_lib()
    counts = [300, 260] if pair_rows else [40, 9]
    E, d, inter = len(counts), 256, 128
    rows = sum(counts)
    x = _rand_bf16((rows, d), 5)
    (gq, gs, dq, ds), _ = _weights_fp8(E, d, inter, seed=6)
    xq, xs = moe.moe_quantize_fp8_rows(x.cuda())
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    shape = _shape(E, d, inter, rows)
    ws = moe.Workspace(moe.moe_expert_ffn_fp8_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_CONTIGUOUS, xq, xs, offsets, 0, gq, gs, dq, ds,
                           ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    bad = gs.clone()
    bad.view(-1)[1] *= 1.5
    moe.moe_expert_ffn_fp8(shape, moe.MOE_LAYOUT_CONTIGUOUS, xq, xs, offsets, 0, gq, bad, dq, ds,
                           ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 1          # MOE_ERR_INVALID_ARG
    assert moe.moe_get_device_status(ws) == 0          # read and cleared


# n_samples: None every token, "tiles" the tokens covering the first and the
# last row of every 128-row m-tile of every expert, else that many sampled
@pytest.mark.parametrize("name,n_samples", [("tiny", None), ("decode", "tiles"), ("few_large", "tiles"),
                                            ("prefill", 2)])
def test_layer_fp8_matches_oracle(name, n_samples):
    ensure_lib()
    cfg = CONFIGS[name]
    t = layer_inputs(name)
    gq, gs = moe.moe_quantize_fp8_blocks(t["w_gate_up"])
    dq, ds = moe.moe_quantize_fp8_blocks(t["w_down"])
    ws = moe.Workspace(moe.moe_layer_fp8_workspace_size(cfg.shape()))
    bias = t["bias"] if cfg.score == SCORE_SIGMOID_BIAS else None
    y = moe.moe_layer_fp8(cfg.shape(), t["x"], t["w_r"], bias, gq, gs, dq, ds, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ids, w = oracle_routing(name)
    if n_samples is None:
        toks = np.arange(cfg.T)
    elif n_samples == "tiles":
        toks, n_tiles = tile_cover_tokens(ids, cfg.E)
        assert tiles_covered(ids, cfg.E, toks) == n_tiles
    else:
        toks = np.sort(np.random.default_rng(2).choice(cfg.T, n_samples, replace=False))
    experts = np.unique(ids[toks])
    # the oracle quantizes what it needs itself: the sampled rows and the
    # weights of the experts they reach
    xq, xs = oracle.quantize_rows_fp8(host_bits(name, "x")[toks])
    wgu, wdn = host_bits(name, "w_gate_up"), host_bits(name, "w_down")
    rgq, rgs = oracle.quantize_blocks_fp8(np.ascontiguousarray(wgu[experts]))
    rdq, rds = oracle.quantize_blocks_fp8(np.ascontiguousarray(wdn[experts]))
    local = {int(e): i for i, e in enumerate(experts)}
    rows_x = np.repeat(np.arange(toks.size), cfg.k)
    row_e = np.array([local[int(e)] for e in ids[toks].ravel()], np.int32)
    yr = oracle.expert_ffn_rows_fp8(xq[rows_x], xs[rows_x], row_e, rgq, rgs, rdq, rds)
    ref = (yr.astype(np.float64).reshape(toks.size, cfg.k, cfg.d) *
           w[toks].astype(np.float64)[:, :, None]).sum(1)
    got = bf16_to_f64(y[torch.from_numpy(toks).cuda().long()])
    check_close(got, ref, bf16_output=True, what=f"{name} fp8 layer")
