"""Device-side error reporting without faulting the GPU: a bounded wait that
runs out records MOE_ERR_TIMEOUT and the context stays usable."""
import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import CONFIGS
from tests.gpu_common import ensure_lib, host_bits, layer_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ensure_lib()
    ws = moe.Workspace(1024)
    moe.moe_selftest_wait_timeout(ws, 2_000_000)  # 2 ms
    assert moe.moe_get_device_status(ws) == 5  # MOE_ERR_TIMEOUT
    assert moe.moe_get_device_status(ws) == 0
    # the context still runs kernels correctly
    cfg = CONFIGS["tiny"]
    t = layer_inputs("tiny")
    ws2 = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    ids, _, _ = moe.moe_route(cfg.shape(), t["x"], t["w_r"], t["bias"], ws2)
    ref, _, _ = oracle.route(host_bits("tiny", "x"), host_bits("tiny", "w_r"),
                             t["bias"].cpu().numpy(), cfg.G, cfg.topk_group, cfg.k, cfg.score)
    assert np.array_equal(ids.cpu().numpy(), ref)


def test_host_side_errors_raise():
    ensure_lib()
    cfg = CONFIGS["tiny"]
    t = layer_inputs("tiny")
    small = moe.Workspace(256)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_layer(cfg.shape(), t["x"], t["w_r"], t["bias"], t["w_gate_up"], t["w_down"],
                      small)
    assert ei.value.status == 3  # MOE_ERR_WORKSPACE
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route(cfg.shape(), t["x"], t["w_r"], None, ws)  # sigmoid needs a bias
    assert ei.value.status == 1
    x_odd = torch.empty(cfg.T * cfg.d + 1, dtype=torch.bfloat16, device="cuda")[1:]
    x_odd = x_odd.view(cfg.T, cfg.d)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route(cfg.shape(), x_odd, t["w_r"], t["bias"], ws)  # misaligned
    assert ei.value.status == 1


def test_reading_an_error_clears_raised_split_flags():
    # A launch that stopped at a timed-out wait can leave split flags of the
    # down GEMM raised.  Plant that state on the host (a status word with
    # the timeout bit, raised flags) and check that reading the status
    # leaves the flags zero for the next launch.
    ensure_lib()
    cfg = CONFIGS["tiny"]
    ws = moe.Workspace(moe.moe_workspace_size(cfg.shape()))
    region = ws.buf[ws.offset:ws.offset + ws.nbytes]
    flags = region[256:256 + 4 * 4096].view(torch.int32)
    flags[::3] = 7
    region[:4].view(torch.int32)[0] = 1 << 5
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 5
    torch.cuda.synchronize()
    assert int(flags.abs().sum()) == 0
    # and a clean word leaves the workspace as it is
    flags[0] = 9
    assert moe.moe_get_device_status(ws) == 0
    assert int(flags[0]) == 9
    flags[0] = 0
