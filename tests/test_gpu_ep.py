"""The expert-parallel layer (dispatch_combine_gb300.ep.moe_layer_ep) on one
GPU as a one-rank NCCL group: every device step (routing, the replicated
dispatch, the masked expert FFN, the combine) and the exchange calls run;
with one rank the exchange returns its input.  The output must match the
oracle layer within the stated tolerance.  The multi-rank exchange logic is
covered on CPU ranks by tests/test_ep_exchange.py."""
import os
import socket

import numpy as np
import pytest
import torch

import dispatch_combine_gb300 as moe
import oracle
from moe_inputs import SCORE_SIGMOID_BIAS, make_tensors_for_shape
from tests.gpu_common import bits, check_close, ensure_lib

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_ep_layer_one_rank_matches_oracle():
    ensure_lib()
    import torch.distributed as dist
    from dispatch_combine_gb300 import ep
    T, d, E, inter, G, tg, k = 384, 1024, 32, 256, 4, 2, 4
    t = make_tensors_for_shape(T, d, E, inter, device="cuda", seed=31, w_std=0.03)
    shape = dict(T=T, d=d, E=E, G=G, topk_group=tg, k=k, inter=inter,
                 score=SCORE_SIGMOID_BIAS, bias_scale=0.15)
    # a placement with copies of the busiest experts (from the planner)
    ws = moe.Workspace(moe.moe_workspace_size(shape))
    ids, _, _ = moe.moe_route(shape, t["x"], t["w_r"], t["bias"], ws)
    load = np.bincount(ids.cpu().numpy().ravel(), minlength=E).astype(np.float64)
    slots, _ = moe.moe_eplb_plan(load, G, 0, 4, E + 8)
    phys = torch.from_numpy(np.asarray(slots, np.int32).reshape(-1)).cuda()
    w_gu = t["w_gate_up"][phys.long()].contiguous()
    w_dn = t["w_down"][phys.long()].contiguous()
    created = False
    if not dist.is_initialized():
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}",
                                rank=0, world_size=1)
        created = True
    try:
        y = ep.moe_layer_ep(shape, t["x"], t["w_r"], t["bias"], phys, w_gu, w_dn)
        torch.cuda.synchronize()
    finally:
        if created:
            dist.destroy_process_group()
    y_ref, _, _ = oracle.layer_tokens(bits(t["x"]), bits(t["w_r"]), t["bias"].cpu().numpy(),
                                      bits(t["w_gate_up"]), bits(t["w_down"]), shape,
                                      np.arange(T, dtype=np.int32))
    check_close(y.float().cpu().numpy(), y_ref, bf16_output=True, what="ep layer")
