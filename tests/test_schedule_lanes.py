"""Persistent schedule: AssignGrid's placement of the backward kernels' work units on
lanes (host only, no GPU).  AugTree paper, Sec. 3.4, Eq. 6: units with work estimates
are placed on a grid of rounds x lanes minimising the largest lane total, exactly for
few units and by largest-first greedy balancing otherwise.

Checked independently of the library's loops: the lanes partition the units; a lane
holds at most ceil(U / L) units in round order; above the exact threshold the placement
is bit-exact with the oracle's largest-first greedy (oracle.assign_grid.lpt) on the
units' weights taken from the exported queue; at or below it the largest lane total
equals the brute-force minimum over all placements (where they can be enumerated; else it
is checked against the greedy and the trivial lower bounds)."""
import numpy as np
import pytest

import shared_prompt_tree_gb300 as at
import workloads as W
from oracle import assign_grid as AG


def units_and_weights(offsets, cfg, op):
    """Unit weights: the costs of the queue's items, one unit per item."""
    q = at.schedule_build(offsets, cfg, op)
    return [int(c) for c in q[:, 5]]


CASES = [
    (W.Tree([300, 129], [[129, 1, 200], [64, 3]]), 8, 2),
    (W.Tree([700], [[300, 20, 5, 128]]), 4, 4),
    (W.Tree([64, 2, 30], [[], [31], [1, 1, 1, 17]]), 6, 2),
    (W.Tree([1300], [[9] * 70 + [650]]), 4, 2),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
@pytest.mark.parametrize("sms", [1, 3, 7, 152])
def test_lanes_are_assign_grid_on_the_queue_costs(ci, sms):
    tree, hq, hkv = CASES[ci]
    cfg = at.make_config(hq, hkv, 128, at.BF16, 0.0, sms, at.KERNEL_TC)
    offs = tree.offsets()
    for op, kid in ((0, at.KID_BWD_QUERY_SIDE), (1, at.KID_BWD_QUERY_SIDE), (2, at.KID_BWD_KEY_SIDE),
                    (3, at.KID_BWD_KEY_SIDE), (4, at.KID_BWD_KEY_SIDE)):
        w = units_and_weights(offs, cfg, op)
        off, units = at.schedule_lanes(offs, cfg, op, kid)
        U = len(w)
        L = min(sms, U)
        assert len(off) == L + 1 and off[0] == 0 and off[-1] == U
        assert sorted(units.tolist()) == list(range(U))
        if U == 0:
            continue
        rounds = -(-U // L)
        assert int(np.max(np.diff(off))) <= rounds
        lane = np.zeros(U, dtype=np.int64)
        rnd = np.zeros(U, dtype=np.int64)
        for l in range(L):
            for r, u in enumerate(units[off[l]:off[l + 1]]):
                lane[u], rnd[u] = l, r
        if U > at.LANES_EXACT_UNITS:
            ref_round, ref_lane = AG.lpt(w, rounds, L)
            assert lane.tolist() == list(ref_lane) and rnd.tolist() == list(ref_round), (op, kid)
        elif L ** U <= 200_000:
            assert AG.makespan(w, lane, L) == AG.brute_force_makespan(w, rounds, L), (op, kid)
        else:
            # Too many placements to enumerate: the exact placement is no worse than the
            # greedy's and no better than the trivial lower bounds.
            mk = AG.makespan(w, lane, L)
            assert mk <= AG.makespan(w, AG.lpt(w, rounds, L)[1], L), (op, kid)
            assert mk >= max(max(w), -(-sum(w) // L)), (op, kid)


def test_lanes_reject_a_kernel_that_does_not_walk_the_queue():
    tree, hq, hkv = CASES[0]
    cfg = at.make_config(hq, hkv, 128, at.BF16, 0.0, 4, at.KERNEL_TC)
    with pytest.raises(at.AugtreeError):
        at.schedule_lanes(tree.offsets(), cfg, 0, at.KID_FWD_TC)  # the forward keeps one block per unit
    with pytest.raises(at.AugtreeError):
        at.schedule_lanes(tree.offsets(), cfg, 2, at.KID_BWD_QUERY_SIDE)
    with pytest.raises(at.AugtreeError):
        at.schedule_lanes(tree.offsets(), cfg, 0, at.KID_BWD_KEY_SIDE)
