"""Pins of the oracle's dispatch onto physical expert copies (reading R15:
the r-th assignment of a logical expert goes to copy r mod n_rep in the
placement's slot order; rows contiguous per physical slot, stable in the
flat assignment index a = t*k + j).  Page: "ep-deploy" handbook, section
"EPLB 与路由约束" (copies of hot experts), and "第十五章" section 4.3 (the
system routes each assignment to one of the expert's equivalent copies,
the less loaded one)."""
import numpy as np
import pytest

import oracle
from moe_inputs import random_ids


def _brute(ids, E, phys):
    """Independent restatement: per assignment its copy by counting earlier
    assignments of the same expert, then a lexicographic sort by (slot, a)."""
    flat = ids.ravel()
    slots_of = {e: [p for p in range(len(phys)) if phys[p] == e] for e in range(E)}
    slot = np.empty(flat.size, np.int64)
    for a, e in enumerate(flat):
        r = int(np.sum(flat[:a] == e))
        slot[a] = slots_of[int(e)][r % len(slots_of[int(e)])]
    order = np.lexsort((np.arange(flat.size), slot))  # by slot, then a
    dest = np.empty(flat.size, np.int64)
    dest[order] = np.arange(flat.size)
    counts = np.bincount(slot, minlength=len(phys))
    src = order // ids.shape[1]
    return counts, dest, src


def _greedy_least_loaded(ids, E, phys):
    """The page's rule taken literally: each assignment, in increasing a,
    goes to the copy of its expert with the fewest rows so far (ties: the
    first copy in slot order)."""
    load = np.zeros(len(phys), np.int64)
    slot = []
    for e in ids.ravel():
        cands = [p for p in range(len(phys)) if phys[p] == e]
        p = min(cands, key=lambda q: (load[q], q))
        load[p] += 1
        slot.append(p)
    return np.array(slot)


@pytest.mark.parametrize("T,k,E,P,seed", [(50, 2, 8, 8, 0), (37, 3, 8, 13, 1), (64, 4, 16, 24, 2),
                                          (1, 1, 4, 9, 3), (120, 8, 32, 48, 4)])
def test_replicated_dispatch_matches_brute_force(T, k, E, P, seed):
    rng = np.random.default_rng(seed)
    ids = random_ids(T, k, E, seed=seed, skew=1.5).numpy()
    # every expert has at least one copy; the extra copies are random, and
    # the slots are shuffled so copies of one expert are not adjacent
    phys = np.concatenate([np.arange(E), rng.integers(0, E, P - E)]).astype(np.int32)
    rng.shuffle(phys)
    counts, offsets, dest, src = oracle.dispatch_replicated(ids, E, phys)
    bc, bd, bs = _brute(ids, E, phys)
    assert np.array_equal(counts, bc)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(bc)]))
    assert np.array_equal(dest, bd)
    assert np.array_equal(src, bs)
    # the rule equals the least-loaded choice of the page
    assert np.array_equal(np.searchsorted(offsets, dest, side="right") - 1,
                          _greedy_least_loaded(ids, E, phys))


def test_one_copy_each_is_the_plain_dispatch():
    ids = random_ids(300, 4, 32, seed=7, skew=2.0).numpy()
    got = oracle.dispatch_replicated(ids, 32, np.arange(32, dtype=np.int32))
    ref = oracle.dispatch(ids, 32)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_copies_of_an_expert_are_balanced():
    ids = random_ids(500, 8, 64, seed=9, skew=2.5).numpy()
    n_e = np.bincount(ids.ravel(), minlength=64)
    phys = np.concatenate([np.arange(64), np.repeat(np.argsort(-n_e)[:16], 2)]).astype(np.int32)
    counts, _, _, _ = oracle.dispatch_replicated(ids, 64, phys)
    for e in range(64):
        c = counts[phys == e]
        assert c.sum() == n_e[e]
        assert c.max() - c.min() <= 1
        assert np.all(np.diff(c) <= 0)  # earlier copies take the larger share


def test_placement_from_the_planner_feeds_the_dispatch():
    # the placement planner's slots (GPU-major) used as the physical order:
    # GPU g's rows are one contiguous range, its count the sum of its slots
    ids = random_ids(2048, 8, 256, seed=3, skew=2.0).numpy()
    load = np.bincount(ids.ravel(), minlength=256).astype(np.float64)
    slots, reps = oracle.eplb_place(load, 8, 4, 32, 288)
    phys = slots.reshape(-1)
    counts, offsets, dest, src = oracle.dispatch_replicated(ids, 256, phys)
    assert counts.sum() == ids.size
    per_gpu = counts.reshape(32, 9).sum(1)
    assert np.array_equal(per_gpu, np.diff(offsets[::9]))
    # copies spread the hot experts: the busiest GPU is close to the mean
    # (the planner's own load figure for the same placement)
    assert per_gpu.max() / per_gpu.mean() < 1.1


def test_rejects_expert_without_copy():
    ids = np.array([[0, 1]], np.int32)
    with pytest.raises(ValueError):
        oracle.dispatch_replicated(ids, 3, np.array([0, 2], np.int32))
