"""GPU expert FFN (tcgen05 grouped GEMMs, SwiGLU fused) against the oracle's
fp64 FFN: contiguous and masked layouts, ragged expert sizes spanning
several 128-row tiles, every N-tile variant, empty experts."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from tests.gpu_common import bits, check_close, ensure_lib

pytestmark = pytest.mark.gpu


def _weights(E, d, inter, seed):
    # g, u ~ N(0, 1) and y of order 1, so that the absolute bound is meaningful
    g = torch.Generator().manual_seed(seed)
    w_gu = (torch.randn(E, 2 * inter, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    w_down = (torch.randn(E, d, inter, generator=g) / inter ** 0.5).to(torch.bfloat16)
    return w_gu, w_down


def check_ffn(got, x_bits, row_e, w_gu_bits, w_down_bits, what):
    """Stated tolerance against the fp64 oracle, plus a much tighter relative
    Frobenius bound against the oracle variant that rounds h to bf16 (the
    GPU's storage format for h): what remains there is only fp32
    accumulation order and the rare bf16 rounding flips of h."""
    ref = oracle.expert_ffn_rows(x_bits, row_e, w_gu_bits, w_down_bits)
    check_close(got, ref, bf16_output=False, what=what)
    ref_hb = oracle.expert_ffn_rows(x_bits, row_e, w_gu_bits, w_down_bits, round_h_bf16=True)
    rel = np.linalg.norm(got - ref_hb) / max(np.linalg.norm(ref_hb), 1e-30)
    assert rel <= 1e-3, f"{what}: rel Frobenius vs h-in-bf16 oracle {rel:.3e}"


def _shape(E, d, inter, T=1, k=1):
    return dict(T=T, d=d, E=E, G=1, topk_group=1, k=k, inter=inter, score=1, bias_scale=0.15)


def _contiguous_case(counts, d, inter, seed):
    E = len(counts)
    rows = int(sum(counts))
    g = torch.Generator().manual_seed(seed + 1)
    x = torch.randn(rows, d, generator=g).to(torch.bfloat16)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    row_e = np.repeat(np.arange(E), counts).astype(np.int32)
    return x, offsets, row_e


@pytest.mark.parametrize("counts,d,inter", [
    ([0, 1, 127, 128, 129, 300], 256, 128),   # gate_up BN=256, down BN=256
    ([5, 0, 0, 260], 512, 64),                # gate_up BN=128 (inter 64)
    ([130, 7], 192, 128),                     # down BN=64
    ([40, 300, 1], 384, 192),                 # down BN=128, gate_up BN=128
    ([3, 200], 4096, 1024),                   # long K in both GEMMs
])
def test_ffn_contiguous(counts, d, inter):
    ensure_lib()
    E = len(counts)
    w_gu, w_down = _weights(E, d, inter, seed=d + inter)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=d)
    rows = x.shape[0]
    shape = _shape(E, d, inter, T=rows, k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x.cuda(), offsets.cuda(), 0,
                           w_gu.cuda(), w_down.cuda(), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    check_ffn(y.cpu().numpy(), bits(x), row_e, bits(w_gu), bits(w_down), "y")


@pytest.mark.parametrize("counts,d,inter", [
    ([1100, 1000], 512, 256),      # ragged pair tiles; the odd CTA of one has no rows
    ([0, 2561, 768], 1024, 384),   # empty expert, exact multiples of 256
    ([4000, 40, 300, 700], 256, 128),
    # last tiles of 1, 16, 17, 100, 128 rows run swapped; 129 and 255 do not
    ([257, 272, 273, 356, 384, 385, 511, 0], 512, 256),
    # swapped tails of 63, 64, 65 rows (N rounded up to 64, 64, 80)
    ([320, 319, 321, 575, 576, 1], 512, 256),
    ([1, 16, 600, 900], 256, 384),  # experts made of one swapped tile
    ([700, 300], 4096, 1024),       # long K
    # down: 15 m-tiles x 16 n-tiles = 240 tiles on 76 pairs, the last 12
    # (swapped tails among them) run as two K halves on two pairs
    ([520, 520, 520, 520, 530], 4096, 256),
    # 192 tiles: a last wave of 40 tiles, not split (80 halves > 76 pairs)
    ([2000, 1000], 4096, 256),
])
def test_ffn_pair_tiles(counts, d, inter):
    # T*k >= 256 rows per expert selects the CTA-pair (cta_group::2) kernels
    ensure_lib()
    E = len(counts)
    assert sum(counts) >= 256 * E
    w_gu, w_down = _weights(E, d, inter, seed=d * 3 + inter)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=d + 7)
    shape = _shape(E, d, inter, T=x.shape[0], k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = torch.full((x.shape[0], d), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x.cuda(), offsets.cuda(), 0,
                       w_gu.cuda(), w_down.cuda(), ws, y_out=y)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    check_ffn(y.cpu().numpy(), bits(x), row_e, bits(w_gu), bits(w_down), "y (pair)")


@pytest.mark.parametrize("counts", [
    [17, 129, 0, 256],     # single-CTA tiles
    [17, 300, 129, 600],   # pair tiles; last tiles of 17, 44 and 88 rows swapped
])
def test_gate_up_alone_matches_oracle_h(counts):
    ensure_lib()
    E, d, inter = 4, 512, 256
    w_gu, w_down = _weights(E, d, inter, seed=3)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=4)
    shape = _shape(E, d, inter, T=x.shape[0], k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    h = moe.moe_expert_gate_up(shape, moe.MOE_LAYOUT_CONTIGUOUS, x.cuda(), offsets.cuda(), 0,
                               w_gu.cuda(), ws)
    _, ref_h = oracle.expert_ffn_rows(bits(x), row_e, bits(w_gu), bits(w_down), return_h=True)
    check_close(h.float().cpu().numpy(), ref_h, bf16_output=True, what="h")
    # down alone on the GPU's own h equals the oracle's down projection of it
    y = moe.moe_expert_down(shape, moe.MOE_LAYOUT_CONTIGUOUS, h, offsets.cuda(), 0,
                            w_down.cuda(), ws)
    hd = h.float().cpu().numpy().astype(np.float64)
    wd = w_down.float().numpy().astype(np.float64)
    ref_y = np.stack([wd[row_e[r]] @ hd[r] for r in range(hd.shape[0])])
    check_close(y.cpu().numpy(), ref_y, bf16_output=False, what="y(down)")
    assert np.abs(y.cpu().numpy() - ref_y).max() < 1e-3


@pytest.mark.parametrize("masked_m,M_max,d,inter,T", [
    ([0, 5, 256, 130], 256, 256, 128, 1),
    ([64, 1, 128], 128, 512, 64, 1),
    # CTA-pair tiles (T*k >= 256 rows per expert, M_max >= 256): full 256-row
    # tiles, a 44-row swapped tail, a 5-row swapped expert, a 200-row plain tail
    ([0, 5, 300, 512, 456], 512, 256, 128, 1280),
])
def test_ffn_masked(masked_m, M_max, d, inter, T):
    ensure_lib()
    E = len(masked_m)
    w_gu, w_down = _weights(E, d, inter, seed=9)
    g = torch.Generator().manual_seed(10)
    x = torch.randn(E, M_max, d, generator=g).to(torch.bfloat16)
    shape = _shape(E, d, inter, T=T)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_MASKED, M_max))
    y = torch.full((E, M_max, d), float("nan"), dtype=torch.float32, device="cuda")
    mm = torch.tensor(masked_m, dtype=torch.int32)
    moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_MASKED, x.cuda(), mm.cuda(), M_max, w_gu.cuda(),
                       w_down.cuda(), ws, y_out=y)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    yh = y.cpu().numpy()
    xb = bits(x)
    for e in range(E):
        m = masked_m[e]
        assert np.all(np.isnan(yh[e, m:])), "rows past masked_m were written"
        if m == 0:
            continue
        check_ffn(yh[e, :m], xb[e, :m], np.full(m, e, np.int32), bits(w_gu), bits(w_down),
                  f"expert {e}")


def test_ffn_masked_overflow_is_flagged_and_clamped():
    ensure_lib()
    E, M_max, d, inter = 2, 128, 256, 128
    w_gu, w_down = _weights(E, d, inter, seed=11)
    x = torch.randn(E, M_max, d, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    shape = _shape(E, d, inter)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_MASKED, M_max))
    mm = torch.tensor([M_max + 50, 3], dtype=torch.int32)
    y = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_MASKED, x.cuda(), mm.cuda(), M_max,
                           w_gu.cuda(), w_down.cuda(), ws)
    assert moe.moe_get_device_status(ws) == 6  # MOE_ERR_OVERFLOW
    check_ffn(y[0].cpu().numpy(), bits(x)[0], np.zeros(M_max, np.int32), bits(w_gu),
              bits(w_down), "clamped expert")


def test_ffn_all_experts_empty_writes_nothing():
    ensure_lib()
    E, d, inter = 3, 256, 128
    w_gu, w_down = _weights(E, d, inter, seed=13)
    shape = _shape(E, d, inter, T=4, k=1)
    x = torch.randn(4, d).to(torch.bfloat16).cuda()
    offsets = torch.zeros(E + 1, dtype=torch.int32).cuda()
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    y = torch.full((4, d), 7.0, dtype=torch.float32, device="cuda")
    moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, x, offsets, 0, w_gu.cuda(),
                       w_down.cuda(), ws, y_out=y)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.all(y == 7.0)


@pytest.mark.parametrize("counts,d,inter", [
    ([300], 512, 256),             # 4 down tiles, all split (2 of them swapped tails)
    ([600, 260, 1], 1024, 512),    # 6 m-tiles x 4 n-tiles, all split (3 swapped tails)
    ([520, 520, 520, 520, 530], 4096, 256),  # 240 tiles, the last 12 split
])
def test_ffn_pair_split_last_wave(counts, d, inter):
    """A short down GEMM runs its last wave as two K halves on two CTA pairs
    (one stores, the other adds after a flag): the result matches the
    oracle, is bit-identical from call to call, and the flags are left
    clear for the next call."""
    ensure_lib()
    E = len(counts)
    w_gu, w_down = _weights(E, d, inter, seed=d + 5 * inter)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=d + 11)
    shape = _shape(E, d, inter, T=x.shape[0], k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    args = (shape, moe.MOE_LAYOUT_CONTIGUOUS, x.cuda(), offsets.cuda(), 0, w_gu.cuda(),
            w_down.cuda(), ws)
    y1 = moe.moe_expert_ffn(*args)
    y2 = moe.moe_expert_ffn(*args)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32)), "split sums not reproducible"
    flags = ws.buf[ws.offset + 256: ws.offset + 256 + 4 * 4096]
    assert int(flags.count_nonzero()) == 0, "split flags left set"
    check_ffn(y1.cpu().numpy(), bits(x), row_e, bits(w_gu), bits(w_down), "y (split)")


def test_ffn_pair_split_beside_a_busy_stream():
    """The split last wave needs no co-residency: with a side stream keeping
    the SMs busy (plain GEMMs that wait on nothing), the split down GEMM
    gives bit-for-bit the result of a run on an idle GPU."""
    ensure_lib()
    counts, d, inter = [520, 520, 520, 520, 530], 4096, 256
    E = len(counts)
    w_gu, w_down = _weights(E, d, inter, seed=d + 5 * inter)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=d + 11)
    shape = _shape(E, d, inter, T=x.shape[0], k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    args = (shape, moe.MOE_LAYOUT_CONTIGUOUS, x.cuda(), offsets.cuda(), 0, w_gu.cuda(),
            w_down.cuda(), ws)
    y_idle = moe.moe_expert_ffn(*args)
    torch.cuda.synchronize()
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    side = torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(side):
            for _ in range(6):
                a = (a @ a) * (1.0 / 64)
        y_busy = moe.moe_expert_ffn(*args)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        assert torch.equal(y_busy.view(torch.int32), y_idle.view(torch.int32))


def test_ffn_pair_split_flags_cleared_by_each_call_and_graph_replays():
    """Every call clears the down GEMM's split flags before the GEMM runs, so
    words left behind (planted here on the host, as an aborted launch could
    leave them) neither disturb the next call nor survive it; and the split
    FFN captured in a CUDA graph gives the eager result on every replay."""
    ensure_lib()
    counts, d, inter = [600, 260, 1], 1024, 512
    E = len(counts)
    w_gu, w_down = _weights(E, d, inter, seed=d + 5 * inter)
    x, offsets, row_e = _contiguous_case(counts, d, inter, seed=d + 11)
    shape = _shape(E, d, inter, T=x.shape[0], k=1)
    ws = moe.Workspace(moe.moe_expert_ffn_workspace_size(shape, moe.MOE_LAYOUT_CONTIGUOUS))
    xd, od, gud, dd = x.cuda(), offsets.cuda(), w_gu.cuda(), w_down.cuda()
    y_ref = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, xd, od, 0, gud, dd, ws)
    torch.cuda.synchronize()
    flags = ws.buf[ws.offset + 256: ws.offset + 256 + 4 * 4096].view(torch.int32)
    flags.fill_(12345)
    y = moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, xd, od, 0, gud, dd, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    assert int(flags.count_nonzero()) == 0, "planted flags survived the call"
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    # the same launches captured once and replayed
    y_g = torch.empty_like(y_ref)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        moe.moe_expert_ffn(shape, moe.MOE_LAYOUT_CONTIGUOUS, xd, od, 0, gud, dd, ws, y_out=y_g,
                           stream=stream)
    for _ in range(3):
        y_g.zero_()
        flags.fill_(12345)
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        assert torch.equal(y_g.view(torch.int32), y_ref.view(torch.int32))
