"""Expert-parallel exchange of the MoE layer (host side).

"第十五章：多节点大模型推理" section 3.4 and the token trace's hop 4 ("分发到两个
专家"): with experts spread over ranks, a dispatch all-to-all carries every
assignment's row to the rank holding its expert, the experts run there, and
a combine all-to-all carries the results back, where the weighted sum is
taken.  "ep-deploy" handbook page, section "EPLB 与路由约束": the ranks hold
physical copies of the logical experts, placed by the planner.

This module plans and performs the two exchanges for one rank of an
expert-parallel group of W ranks, each holding S = P / W consecutive
physical slots of the placement (GPU-major, as moe_eplb_plan returns them).
The send side is the replicated dispatch of the rank's own tokens
(moe_dispatch_replicated, or anything with its layout): rows contiguous per
physical slot in slot order, so the rows for rank q are one contiguous
range.  The exchange itself is torch.distributed all_to_all_single on the
group (NCCL for device tensors, gloo for host tensors).

Receive layout.  Rows arrive ordered by (source rank, local slot, source
order).  Each local slot s gets the masked layout of the expert FFN: rows
[0, masked_m[s]) of slab s in (source rank, source order) order, M_max rows
per slab (masked_m rounded up to 128).  The return exchange sends every
result row back in the order it arrived, so each source gets its rows in
its own send order and combines them with its dispatch's dest.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.distributed as dist

TILE_ROWS = 128


@dataclass
class EPPlan:
    """The exchange plan of one rank (all sizes host ints)."""
    world: int
    rank: int
    slots_per_rank: int
    send_splits: list          # rows sent to each rank
    recv_counts: torch.Tensor  # [W, S] rows from rank q for local slot s (int64, host)
    recv_splits: list          # rows received from each rank
    masked_m: torch.Tensor     # [S] rows of each local slot (int64, host)
    M_max: int                 # slab height of the masked layout
    masked_index: torch.Tensor  # [rows received] slab row (s * M_max + i) of each received row

    @property
    def rows_received(self) -> int:
        return int(sum(self.recv_splits))


def plan_exchange(counts_phys: torch.Tensor, slots_per_rank: int, group=None) -> EPPlan:
    """Exchange the per-slot row counts of this rank's send side and derive
    the plan.  counts_phys [P] (P = W * slots_per_rank) are this rank's rows
    per physical slot (any device; copied to the host)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    S = int(slots_per_rank)
    # the counts travel on their own device (NCCL exchanges device tensors,
    # gloo host ones); the plan's arithmetic is done on the host
    dev_counts = counts_phys.detach().to(torch.int64).reshape(-1).contiguous()
    if dev_counts.numel() != world * S:
        raise ValueError(f"counts_phys has {dev_counts.numel()} slots, expected {world} x {S}")
    counts = dev_counts.cpu()
    send_splits = [int(v) for v in counts.view(world, S).sum(1)]
    # rank q's counts for my slots arrive as block q of recv
    recv = torch.empty_like(dev_counts)
    dist.all_to_all_single(recv, dev_counts, group=group)
    recv_counts = recv.cpu().view(world, S)
    recv_splits = [int(v) for v in recv_counts.sum(1)]
    masked_m = recv_counts.sum(0)
    m = int(masked_m.max()) if S > 0 else 0
    M_max = max(TILE_ROWS, (m + TILE_ROWS - 1) // TILE_ROWS * TILE_ROWS)
    # received row (q, s, i) -> slab row s * M_max + (rows of slot s from
    # ranks before q) + i
    before = torch.cumsum(recv_counts, 0) - recv_counts       # [W, S]
    flat = recv_counts.reshape(-1)                              # (q, s) blocks in arrival order
    first_row = torch.cumsum(flat, 0) - flat                    # arrival index of each block's row 0
    i_in_block = torch.arange(int(flat.sum())) - first_row.repeat_interleave(flat)
    base = torch.arange(S).repeat(world) * M_max + before.reshape(-1)
    masked_index = base.repeat_interleave(flat) + i_in_block
    return EPPlan(world, rank, S, send_splits, recv_counts, recv_splits, masked_m, M_max,
                  masked_index)


def exchange_rows(send: torch.Tensor, plan: EPPlan, group=None) -> torch.Tensor:
    """Dispatch exchange: rows of this rank's send side (ordered by physical
    slot) to the ranks holding the slots; returns the received rows in
    arrival order [(source rank, local slot, source order)]."""
    recv = torch.empty((plan.rows_received,) + tuple(send.shape[1:]), dtype=send.dtype,
                       device=send.device)
    dist.all_to_all_single(recv, send.contiguous(), output_split_sizes=plan.recv_splits,
                           input_split_sizes=plan.send_splits, group=group)
    return recv


def to_masked(recv: torch.Tensor, plan: EPPlan) -> torch.Tensor:
    """Received rows -> masked layout [S, M_max, ...] (rows past masked_m are
    zero)."""
    out = torch.zeros((plan.slots_per_rank * plan.M_max,) + tuple(recv.shape[1:]),
                      dtype=recv.dtype, device=recv.device)
    out.index_copy_(0, plan.masked_index.to(recv.device), recv)
    return out.view((plan.slots_per_rank, plan.M_max) + tuple(recv.shape[1:]))


def from_masked(y_masked: torch.Tensor, plan: EPPlan) -> torch.Tensor:
    """Result rows of the masked layout back in arrival order."""
    flat = y_masked.reshape((plan.slots_per_rank * plan.M_max,) + tuple(y_masked.shape[2:]))
    return flat.index_select(0, plan.masked_index.to(flat.device))


def return_rows(y_recv: torch.Tensor, plan: EPPlan, group=None) -> torch.Tensor:
    """Combine exchange: result rows (in arrival order) back to their source
    ranks; returns this rank's rows in its own send order (physical slot
    order), ready for the combine with its dispatch's dest."""
    out = torch.empty((int(sum(plan.send_splits)),) + tuple(y_recv.shape[1:]),
                      dtype=y_recv.dtype, device=y_recv.device)
    dist.all_to_all_single(out, y_recv.contiguous(), output_split_sizes=plan.send_splits,
                           input_split_sizes=plan.recv_splits, group=group)
    return out


def moe_layer_ep(shape, x, w_r, bias, phys_expert, w_gate_up_local, w_down_local, group=None,
                 stream=None):
    """One rank's MoE layer with expert parallelism: its tokens x [T, d] are
    routed and dispatched onto the placement's physical slots
    (phys_expert [P], the same on every rank), rows travel to the ranks
    holding the slots, each rank runs its S = P / W slots' experts
    (w_gate_up_local [S, 2*inter, d], w_down_local [S, d, inter]: the
    weights of the logical experts its slots hold) on the masked layout, the
    results travel back and the rank combines its tokens.  Every compute
    step is a kernel of libmoe.so; the exchanges are all_to_all_single on
    `group`, the two row permutations around the expert FFN index_copy /
    index_select on the device.  Returns y [T, d] bf16."""
    from . import _lib as moe
    world = dist.get_world_size(group)
    P = int(phys_expert.numel())
    if P % world:
        raise ValueError("the physical slots must split evenly over the ranks")
    S = P // world
    s = moe.as_shape(shape)
    ws = moe.Workspace(moe.moe_workspace_size(shape), device=x.device)
    ids, w, _ = moe.moe_route(shape, x, w_r, bias, ws, stream=stream)
    rws = moe.Workspace(moe.moe_dispatch_replicated_workspace_size(shape, P), device=x.device)
    counts, offsets, src, dest, x_send = moe.moe_dispatch_replicated(shape, phys_expert, ids,
                                                                     x, rws, stream=stream)
    plan = plan_exchange(counts, S, group)
    x_masked = to_masked(exchange_rows(x_send, plan, group), plan)
    fshape = dict(T=1, d=s.d, E=S, G=1, topk_group=1, k=1, inter=s.inter, score=1,
                  bias_scale=0.15)
    fws = moe.Workspace(moe.moe_expert_ffn_workspace_size(fshape, moe.MOE_LAYOUT_MASKED,
                                                          plan.M_max), device=x.device)
    masked_m = plan.masked_m.to(device=x.device, dtype=torch.int32)
    y_masked = moe.moe_expert_ffn(fshape, moe.MOE_LAYOUT_MASKED, x_masked, masked_m, plan.M_max,
                                  w_gate_up_local, w_down_local, fws, stream=stream)
    y_phys = return_rows(from_masked(y_masked, plan), plan, group)
    y = moe.moe_combine(shape, y_phys, dest, w, stream=stream)
    for wsx in (ws, rws, fws):
        st = moe.moe_get_device_status(wsx)
        if st != 0:
            raise moe.MoEError("moe_layer_ep", st)
    return y
