"""Expert-parallel exchange plan and all-to-all (dispatch_combine_gb300.ep)
with two gloo ranks on CPU: each rank dispatches its own tokens onto the
placement's physical copies (the oracle's replicated dispatch stands in for
the GPU kernel), the rows travel to the ranks holding their slots, each
rank runs its slots' experts on the masked layout, the results travel back
and each rank combines its tokens.  The outputs must equal the
single-process oracle layer's for every token, bit for bit; the plan's
receive counts must add up to the global assignment counts per expert.
Pages: "第十五章" section 3.4 (dispatch / combine all-to-all), the token
trace's hop 4, and "ep-deploy" section "EPLB 与路由约束" (placement)."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

W = 2                 # ranks
T_LOCAL = 40          # tokens per rank
E, K, D, INTER = 8, 2, 64, 32
S = 6                 # physical slots per rank (P = 12: 4 extra copies)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    """Seeded global problem: bf16 bit patterns of x and the expert weights,
    routing ids and combine weights of all W * T_LOCAL tokens, placement."""
    from moe_inputs import random_ids, random_weights
    import torch
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(W * T_LOCAL, D, generator=g)).to(torch.bfloat16)
    w_gu = (torch.randn(E, 2 * INTER, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    w_dn = (torch.randn(E, D, INTER, generator=g) / INTER ** 0.5).to(torch.bfloat16)
    ids = random_ids(W * T_LOCAL, K, E, seed=6, skew=1.5).numpy()
    w = random_weights(W * T_LOCAL, K, seed=7).numpy().astype(np.float32)
    phys = np.array([0, 1, 2, 3, 0, 4, 5, 6, 7, 1, 0, 2], np.int32)  # copies of 0 (3), 1, 2
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return bits(x), bits(w_gu), bits(w_dn), ids, w, phys


def _rank_main(rank, port, q):
    try:
        _rank_body(rank, port, q)
    except Exception as e:  # report instead of leaving the other rank waiting
        q.put((rank, repr(e), None, None, None, None))
        raise


def _rank_body(rank, port, q):
    import torch
    import torch.distributed as dist
    import oracle
    from dispatch_combine_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(W))
    import datetime
    dist.init_process_group("gloo", rank=rank, world_size=W,
                            timeout=datetime.timedelta(seconds=60))
    xb, gub, dnb, ids, w, phys = _problem()
    tok = slice(rank * T_LOCAL, (rank + 1) * T_LOCAL)
    # send side: this rank's tokens onto the physical copies
    counts, offsets, dest, src = oracle.dispatch_replicated(ids[tok], E, phys)
    # bf16 bit patterns travel as int32 (gloo has no 16-bit integer type)
    x_send = torch.from_numpy(xb[tok][src].astype(np.int32))
    plan = ep.plan_exchange(torch.from_numpy(counts), S)
    x_recv = ep.exchange_rows(x_send, plan)
    x_masked = ep.to_masked(x_recv, plan).numpy().astype(np.uint16)   # [S, M_max, D]
    # the experts of this rank's slots, on the masked rows
    y_masked = np.zeros((S, plan.M_max, D))
    for s in range(S):
        m = int(plan.masked_m[s])
        if m:
            e = int(phys[rank * S + s])
            y_masked[s, :m] = oracle.expert_ffn_rows(x_masked[s, :m], np.full(m, e, np.int32),
                                                     gub, dnb)
    y_recv = ep.from_masked(torch.from_numpy(y_masked), plan)
    y_phys = ep.return_rows(y_recv, plan).numpy()
    y = oracle.combine(y_phys, dest, w[tok], T_LOCAL, K)
    q.put((rank, y, plan.recv_counts.numpy(), plan.masked_m.numpy(), plan.send_splits,
           plan.recv_splits))
    dist.destroy_process_group()


def test_ep_exchange_two_gloo_ranks_matches_single_process():
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(W)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
    for r in out:
        assert not isinstance(r[1], str), f"rank {r[0]} failed: {r[1]}"
    for p in procs:
        assert p.exitcode == 0
    xb, gub, dnb, ids, w, phys = _problem()
    # single process: the whole batch, logical dispatch, experts, combine
    counts, offsets, dest, src = oracle.dispatch(ids, E)
    y_perm = oracle.expert_ffn_rows(xb[src], np.repeat(np.arange(E), counts).astype(np.int32),
                                    gub, dnb)
    y_ref = oracle.combine(y_perm, dest, w, W * T_LOCAL, K)
    for rank, y, recv_counts, masked_m, send_splits, recv_splits in out:
        assert np.array_equal(y, y_ref[rank * T_LOCAL:(rank + 1) * T_LOCAL]), rank
        # what rank r received from q is what q sent to r
        assert recv_splits == [out[qq][4][rank] for qq in range(W)]
    # every assignment reached exactly one copy of its expert
    got = np.zeros(E, np.int64)
    for rank, _, _, masked_m, _, _ in out:
        for s in range(S):
            got[phys[rank * S + s]] += masked_m[s]
    assert np.array_equal(got, np.bincount(ids.ravel(), minlength=E))
