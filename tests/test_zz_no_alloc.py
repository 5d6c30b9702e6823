"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a runtime that reserves all of HBM up front, plain C
callers without a device allocator, paths where cudaMalloc is not allowed).
Its scratch lives in a fixed array inside the library instead of a caller
workspace.  It must give exactly the results of moe_dispatch, call after
call, although every call reuses the same array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import random_ids
from tests.gpu_common import bits, ensure_lib

pytestmark = pytest.mark.gpu


def _shape(T, d, E, k):
    return dict(T=T, d=d, E=E, G=1, topk_group=1, k=k, inter=64, score=1, bias_scale=0.15)


def _case(T, k, E, d, seed, skew):
    ids = random_ids(T, k, E, seed=seed, skew=skew).cuda()
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return ids, x.cuda()


def _check_against_oracle(ids, x, E, got):
    """counts, offsets, dest and src_token equal the oracle's stable counting
    sort; every gathered row is its source token's row, bit for bit."""
    counts, offsets, dest, src = oracle.dispatch(ids.cpu().numpy(), E)
    for name, ref, g in zip(["counts", "offsets", "src_token", "dest"],
                            [counts, offsets, src, dest], got[:4]):
        assert np.array_equal(g.cpu().numpy(), ref), name
    if x is not None:
        assert np.array_equal(bits(got[4]), bits(x)[src])


@pytest.mark.parametrize("cases", [
    # 128 assignments per chunk (T*k <= 32768)
    [(1000, 8, 256, 136, 11, 2.0), (513, 4, 5, 24, 12, 0.0)],
    # 512 assignments per chunk (T*k > 32768), then a small call after it
    [(8192, 8, 256, 64, 13, 1.5), (100, 2, 16, 32, 14, 0.0)],
])
def test_noalloc_dispatch_equals_workspace_dispatch_twice(cases):
    ensure_lib()
    # two calls in a row with different routings: the second call reuses the
    # array the first one filled and must not see its leftovers
    for T, k, E, d, seed, skew in cases:
        shape = _shape(T, d, E, k)
        ids, x = _case(T, k, E, d, seed, skew)
        ws = moe.Workspace(moe.moe_workspace_size(shape))
        ref = moe.moe_dispatch(shape, ids, x, ws)
        got = moe.moe_dispatch_noalloc(shape, ids, x)
        torch.cuda.synchronize()
        for name, r, g in zip(["counts", "offsets", "src_token", "dest"], ref[:4], got[:4]):
            assert torch.equal(r, g), name
        assert np.array_equal(bits(ref[4]), bits(got[4]))
        _check_against_oracle(ids, x, E, got)


def test_noalloc_dispatch_at_its_largest_shape():
    ensure_lib()
    # ceil(T*k/512) * E = 1024 * 256 = 262144 entries: the whole array
    T, k, E, d = 65536, 8, 256, 16
    shape = _shape(T, d, E, k)
    ids, x = _case(T, k, E, d, 15, 1.0)
    got = moe.moe_dispatch_noalloc(shape, ids, x)
    torch.cuda.synchronize()
    _check_against_oracle(ids, x, E, got)


def test_noalloc_dispatch_rejects_shapes_beyond_its_array():
    ensure_lib()
    # ceil(T*k/512) * E = 1025 * 256 > 262144 entries (512 per chunk above 32768)
    T, k, E = 65600, 8, 256
    shape = _shape(T, 8, E, k)
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_dispatch_noalloc(shape, ids, None)
    assert ei.value.status == 2  # MOE_ERR_UNSUPPORTED
