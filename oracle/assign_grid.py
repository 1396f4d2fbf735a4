"""Reference AssignGrid: placement of replay units on replay rounds x replay lanes.

TEST INFRASTRUCTURE ONLY: imported by tests, never by the library.

AugTree paper, Sec. 3.4 ("Replay units and grid assignment", Eq. 6): a unit k with work
estimate w_k is placed on a cell (round, lane) of a b x s grid; the objective is the
replay critical path, the largest lane total max_j sum_{k on lane j} w_k.  Each cell
holds one unit, so a lane takes at most b units (the reading of the grid in which the
round count b constrains the placement).  The pages solve the problem exactly for
small unit counts and by largest-first greedy balancing otherwise.

brute_force_makespan is the definition of the minimum written out: every placement of
every unit on every lane, kept if no lane exceeds b units.  lpt is the greedy with the
library's tie rules (weight descending then index ascending; the least loaded lane
with a free round, the lowest lane on ties), in plain loops.
"""
from __future__ import annotations

import itertools
from typing import List, Sequence, Tuple


def lane_totals(w: Sequence[int], lane: Sequence[int], lanes: int) -> List[int]:
    tot = [0] * lanes
    for k, j in enumerate(lane):
        tot[j] += int(w[k])
    return tot


def makespan(w: Sequence[int], lane: Sequence[int], lanes: int) -> int:
    return max(lane_totals(w, lane, lanes)) if len(w) else 0


def brute_force_makespan(w: Sequence[int], rounds: int, lanes: int) -> int:
    """Minimum over all placements (lanes ** U of them: tiny inputs only)."""
    best = None
    for lane in itertools.product(range(lanes), repeat=len(w)):
        counts = [0] * lanes
        for j in lane:
            counts[j] += 1
        if max(counts, default=0) > rounds:
            continue
        m = makespan(w, lane, lanes)
        if best is None or m < best:
            best = m
    if best is None:
        raise ValueError("no placement: more units than cells")
    return best


def largest_first(w: Sequence[int]) -> List[int]:
    return sorted(range(len(w)), key=lambda k: (-int(w[k]), k))


def rounds_in_lanes(w: Sequence[int], lane: Sequence[int], lanes: int) -> List[int]:
    """Within each lane the units take rounds 0, 1, ... in largest-first order."""
    used = [0] * lanes
    rnd = [0] * len(w)
    for k in largest_first(w):
        rnd[k] = used[lane[k]]
        used[lane[k]] += 1
    return rnd


def lpt(w: Sequence[int], rounds: int, lanes: int) -> Tuple[List[int], List[int]]:
    """Largest-first greedy placement: (round, lane) per unit."""
    load = [0] * lanes
    used = [0] * lanes
    lane = [0] * len(w)
    for k in largest_first(w):
        best = None
        for j in range(lanes):
            if used[j] < rounds and (best is None or load[j] < load[best]):
                best = j
        if best is None:
            raise ValueError("no placement: more units than cells")
        lane[k] = best
        load[best] += int(w[k])
        used[best] += 1
    return rounds_in_lanes(w, lane, lanes), lane
