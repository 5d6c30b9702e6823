"""Oracle pins for the expert placement of the "ep-deploy" handbook page,
section "EPLB 与路由约束": global and hierarchical placement of the page's
routing simulation reproduce its printed busiest/mean GPU load and nodes per
token (fixture tests/golden/ep_deploy_routing_sim.txt), plus invariants of
the greedy steps on random loads."""
import numpy as np
import pytest

import oracle
from tests.test_oracle_router import _golden_rows, page_sim_scores


def _page_load():
    ids = oracle.select(page_sim_scores(), G=8, topk_group=4, k=8, group_sum_f32=False)
    return ids, np.bincount(ids.ravel(), minlength=256).astype(np.float64)


def placement_report(ids, load, gpu_slots, nodes):
    """The page's two statistics for a placement: busiest GPU load over the
    mean (each replica takes load / replicas), and the mean number of nodes
    a token's 8 experts reach over the first 2000 tokens, a replica on a node
    the token already reaches being preferred, else the lowest node."""
    gpus = gpu_slots.shape[0]
    reps = np.zeros(load.size, int)
    for row in gpu_slots:
        for e in row:
            reps[e] += 1
    gpu_load = [sum(load[e] / reps[e] for e in row) for row in gpu_slots]
    ratio = max(gpu_load) / float(np.mean(gpu_load))
    where = {}
    for g, row in enumerate(gpu_slots):
        for e in row:
            where.setdefault(int(e), set()).add(g // (gpus // nodes))
    touched = []
    for r in ids[:2000]:
        reached = set()
        for e in r:
            if not (where[int(e)] & reached):
                reached.add(min(where[int(e)]))
        touched.append(len(reached))
    return f"{ratio:.2f}", f"{float(np.mean(touched)):.2f}"


@pytest.mark.parametrize("place", ["global", "hier"])
def test_eplb_reproduces_page_printed_results(place):
    ids, load = _page_load()
    checked = 0
    for nodes, gpus, pl, ratio, ntok in _golden_rows():
        if pl != place:
            continue
        phys = {(4, 32): 288, (8, 64): 320}[(nodes, gpus)]
        slots, reps = oracle.eplb_place(load, 8, nodes if place == "hier" else 0, gpus, phys)
        assert reps.sum() == phys and (reps >= 1).all()
        got = placement_report(ids, load, slots, nodes)
        assert got == (ratio, ntok), (nodes, gpus, place, got, ratio, ntok)
        checked += 1
    assert checked == 2


@pytest.mark.parametrize("E,groups,nodes,gpus,phys,seed", [
    (256, 8, 4, 32, 288, 1), (256, 8, 0, 64, 320, 2), (64, 8, 2, 8, 80, 3),
    (16, 4, 4, 4, 16, 4), (32, 4, 0, 4, 48, 5)])
def test_eplb_invariants(E, groups, nodes, gpus, phys, seed):
    g = np.random.default_rng(seed)
    load = np.round(g.gamma(1.0, 100.0, E))          # integer loads with ties
    slots, reps = oracle.eplb_place(load, groups, nodes, gpus, phys)
    assert slots.shape == (gpus, phys // gpus)
    assert np.array_equal(np.bincount(slots.ravel(), minlength=E), reps)
    assert (reps >= 1).all() and reps.sum() == phys
    if nodes:
        # every expert's replicas stay in its group's node, groups stay whole
        per_node = gpus // nodes
        gsize = E // groups
        for e in range(E):
            homes = {gi // per_node for gi in range(gpus) if e in slots[gi]}
            assert len(homes) == 1
        for grp in range(groups):
            homes = {gi // per_node for gi in range(gpus)
                     for e in range(grp * gsize, (grp + 1) * gsize) if e in slots[gi]}
            assert len(homes) == 1
    # replication: no expert could give a replica to another and lower the
    # largest load per replica (greedy optimality of the max)
    per_rep = load / reps
    if nodes == 0:
        worst = per_rep.max()
        for e in range(E):
            if reps[e] > 1:
                assert load[e] / (reps[e] - 1) >= worst - 1e-9


def test_eplb_no_replicas_one_expert_per_gpu_is_a_permutation():
    load = np.arange(16, dtype=np.float64)
    slots, reps = oracle.eplb_place(load, 4, 0, 16, 16)
    assert sorted(slots.ravel().tolist()) == list(range(16)) and (reps == 1).all()
    # heaviest first into the lightest empty GPU: GPU i gets expert 15 - i
    assert slots.ravel().tolist() == list(range(15, -1, -1))
