"""The library's expert placement planner (moe_eplb_plan, host C++ behind the
C ABI; no GPU) against the oracle placement, and against the printed results
of the "ep-deploy" handbook page's placement simulation."""
import numpy as np
import pytest

import dispatch_combine_gb300 as moe
import oracle
from tests.gpu_common import ensure_lib
from tests.test_oracle_eplb import _page_load, placement_report
from tests.test_oracle_router import _golden_rows


@pytest.mark.parametrize("place", ["global", "hier"])
def test_planner_reproduces_page_printed_results(place):
    ensure_lib()
    ids, load = _page_load()
    checked = 0
    for nodes, gpus, pl, ratio, ntok in _golden_rows():
        if pl != place:
            continue
        phys = {(4, 32): 288, (8, 64): 320}[(nodes, gpus)]
        slots, reps = moe.moe_eplb_plan(load, 8, nodes if place == "hier" else 0, gpus, phys)
        assert placement_report(ids, load, slots, nodes) == (ratio, ntok)
        checked += 1
    assert checked == 2


@pytest.mark.parametrize("E,groups,nodes,gpus,phys", [
    (256, 8, 4, 32, 288), (256, 8, 8, 64, 320), (256, 8, 0, 64, 320), (64, 8, 2, 8, 80),
    (16, 4, 4, 4, 16), (32, 4, 0, 4, 48), (128, 16, 4, 16, 160), (8, 1, 0, 2, 12)])
def test_planner_matches_oracle(E, groups, nodes, gpus, phys):
    ensure_lib()
    g = np.random.default_rng(E + phys)
    for trial in range(20):
        if trial % 3 == 0:
            load = np.round(g.gamma(0.7, 50.0, E))       # integers: many ties
        elif trial % 3 == 1:
            load = g.random(E) * 1000.0
        else:
            load = np.ones(E)                              # all equal
        s1, r1 = moe.moe_eplb_plan(load, groups, nodes, gpus, phys)
        s2, r2 = oracle.eplb_place(load, groups, nodes, gpus, phys)
        assert np.array_equal(s1, s2) and np.array_equal(r1, r2), trial


def test_planner_rejects_bad_sizes():
    ensure_lib()
    load = np.ones(256)
    for args in [(7, 4, 32, 288), (8, 3, 32, 288), (8, 4, 30, 288), (8, 4, 32, 250),
                 (8, 4, 32, 300)]:
        with pytest.raises(moe.MoEError):
            moe.moe_eplb_plan(load, *args)
    with pytest.raises(moe.MoEError):
        moe.moe_eplb_plan(-np.ones(256), 8, 4, 32, 288)
