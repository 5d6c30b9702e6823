"""GPU dispatch (bit-exact against the oracle's stable counting sort) and
combine (identity experts return x exactly; random inputs within bf16
rounding of the fp64 oracle)."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import random_ids, random_weights
from tests.gpu_common import bits, ensure_lib, half_ulp_bf16

pytestmark = pytest.mark.gpu


def _shape(T, d, E, k):
    G = 1
    return dict(T=T, d=d, E=E, G=G, topk_group=1, k=k, inter=64, score=1, bias_scale=0.15)


@pytest.mark.parametrize("T,k,E,d,skew", [
    (1, 1, 1, 8, 0.0),
    (1, 8, 256, 64, 0.0),
    (64, 2, 16, 256, 0.0),
    (1000, 8, 256, 136, 2.0),    # 8000 assignments: 15 full chunks + ragged tail
    (4096, 8, 256, 7168, 1.5),
    (16384, 8, 256, 512, 2.5),   # 131072 assignments, hot experts
    (3000, 3, 1024, 64, 3.0),
    (513, 4, 5, 24, 0.0),
])
def test_dispatch_bit_exact(T, k, E, d, skew):
    ensure_lib()
    ids = random_ids(T, k, E, seed=T * 7 + E, skew=skew)
    x = (torch.randn(T, d, generator=torch.Generator().manual_seed(T)) * 1.0).to(torch.bfloat16)
    shape = _shape(T, d, E, k)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    counts, offsets, src, dest, x_perm = moe.moe_dispatch(shape, ids.cuda(), x.cuda(), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    r_counts, r_offsets, r_dest, r_src = oracle.dispatch(ids.numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), r_counts)
    assert np.array_equal(offsets.cpu().numpy(), r_offsets)
    assert np.array_equal(dest.cpu().numpy(), r_dest)
    assert np.array_equal(src.cpu().numpy(), r_src)
    assert np.array_equal(bits(x_perm), bits(x)[r_src])


def test_dispatch_all_to_one_expert_and_indices_only():
    ensure_lib()
    T, k, E = 2000, 4, 64
    ids = torch.zeros(T, k, dtype=torch.int32)
    ids[:, 1:] = torch.arange(1, k, dtype=torch.int32)
    shape = _shape(T, 64, E, k)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    counts, offsets, src, dest, x_perm = moe.moe_dispatch(shape, ids.cuda(), None, ws)
    assert x_perm is None
    r_counts, r_offsets, r_dest, r_src = oracle.dispatch(ids.numpy(), E)
    assert np.array_equal(dest.cpu().numpy(), r_dest)
    assert np.array_equal(src.cpu().numpy(), r_src)
    assert np.array_equal(counts.cpu().numpy(), r_counts)


def test_dispatch_flags_out_of_range_ids():
    ensure_lib()
    T, k, E = 100, 2, 16
    ids = random_ids(T, k, E, seed=1)
    ids[5, 1] = 99
    ids[70, 0] = -3
    shape = _shape(T, 64, E, k)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    x = torch.zeros(T, 64, dtype=torch.bfloat16, device="cuda")
    counts, offsets, _, _, _ = moe.moe_dispatch(shape, ids.cuda(), x, ws)
    assert moe.moe_get_device_status(ws) == 1  # MOE_ERR_INVALID_ARG
    assert int(counts.sum()) == T * k - 2
    assert moe.moe_get_device_status(ws) == 0  # cleared by the read


def test_combine_identity_experts_return_x_exactly():
    ensure_lib()
    T, k, E, d = 777, 8, 256, 512
    ids = random_ids(T, k, E, seed=5, skew=1.0)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    shape = _shape(T, d, E, k)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    _, _, _, dest, x_perm = moe.moe_dispatch(shape, ids.cuda(), x.cuda(), ws)
    w = random_weights(T, k, seed=2)
    w = (w / w.sum(1, keepdim=True)).float().cuda()
    y = moe.moe_combine(shape, x_perm.float().contiguous(), dest, w)
    assert np.array_equal(bits(y), bits(x))


@pytest.mark.parametrize("T,k,d", [(1, 1, 8), (300, 8, 7168), (2048, 2, 4096), (65, 3, 40)])
def test_combine_matches_oracle(T, k, d):
    ensure_lib()
    n = T * k
    g = torch.Generator().manual_seed(n + d)
    y_perm = torch.randn(n, d, generator=g) * 3
    dest = torch.randperm(n, generator=g).to(torch.int32)
    w = random_weights(T, k, seed=d)
    shape = _shape(T, d, max(k, 1), k)
    y = moe.moe_combine(shape, y_perm.cuda(), dest.cuda(), w.cuda())
    ref = oracle.combine(y_perm.numpy(), dest.numpy(), w.numpy(), T, k)
    # fp32 accumulation error scales with sum_j |w_j y_j| (cancellation), then
    # one bf16 rounding of the result
    mag = oracle.combine(np.abs(y_perm.numpy()), dest.numpy(), np.abs(w.numpy()), T, k)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= half_ulp_bf16(ref) + k * 2.0 ** -23 * mag + 1e-30)
