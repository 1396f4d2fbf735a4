"""AssignGrid (AugTree paper, Sec. 3.4, Eq. 6): the library's placement planner against
the oracle, and the oracle against published values.  Host only (no GPU)."""
import numpy as np
import pytest

from oracle import assign_grid as ref


# ---------------------------------------------------------------- oracle pins
def test_oracle_graham_tight_example():
    # Graham (1969), the tight case of the 4/3 - 1/(3m) bound for largest-first list
    # scheduling on m = 3 machines: jobs 5,5,4,4,3,3,3; optimum 9 (5+4, 5+4, 3+3+3),
    # largest-first 11.
    w = [5, 5, 4, 4, 3, 3, 3]
    assert ref.brute_force_makespan(w, rounds=7, lanes=3) == 9
    rnd, lane = ref.lpt(w, rounds=7, lanes=3)
    assert ref.makespan(w, lane, 3) == 11
    assert 11 / 9 == pytest.approx(4 / 3 - 1 / 9)


def test_oracle_two_machine_example():
    # 3,3,2,2,2 on two machines: optimum 6 (3+3 | 2+2+2); largest-first puts one 3
    # with two 2s (7).
    w = [3, 3, 2, 2, 2]
    assert ref.brute_force_makespan(w, rounds=5, lanes=2) == 6
    assert ref.makespan(w, ref.lpt(w, 5, 2)[1], 2) == 7


def test_oracle_closed_forms():
    rng = np.random.default_rng(1)
    for _ in range(20):
        u = int(rng.integers(1, 6))
        w = [int(x) for x in rng.integers(0, 50, u)]
        # As many lanes as units: every unit alone, the makespan is the largest unit.
        assert ref.brute_force_makespan(w, rounds=1, lanes=u) == max(w)
        # One lane: everything in sequence.
        assert ref.brute_force_makespan(w, rounds=u, lanes=1) == sum(w)
    # Equal weights: ceil(U / s) units on the fullest lane.
    for u, s in [(7, 3), (8, 4), (5, 2)]:
        assert ref.brute_force_makespan([10] * u, rounds=u, lanes=s) == 10 * -(-u // s)
    # The round count binds: with one round per lane the big units cannot share a lane.
    assert ref.brute_force_makespan([9, 1, 1, 1], rounds=2, lanes=2) == 10
    assert ref.brute_force_makespan([9, 1, 1, 1], rounds=3, lanes=2) == 9


def test_oracle_rounds_in_lanes():
    w = [4, 9, 4, 1]
    lane = [0, 0, 0, 1]
    # Lane 0 holds 9 (unit 1), 4 (unit 0), 4 (unit 2): largest first, ties by index.
    assert ref.rounds_in_lanes(w, lane, 2) == [1, 0, 2, 0]


# ---------------------------------------------------------------- library vs oracle
def _valid(w, rnd, lane, rounds, lanes):
    cells = set()
    for k in range(len(w)):
        assert 0 <= lane[k] < lanes and 0 <= rnd[k] < rounds
        assert (rnd[k], lane[k]) not in cells
        cells.add((rnd[k], lane[k]))
    assert list(rnd) == ref.rounds_in_lanes(w, list(lane), lanes)


def test_exact_matches_brute_force(augtree_lib):
    import shared_prompt_tree_gb300 as at
    rng = np.random.default_rng(7)
    for _ in range(150):
        u = int(rng.integers(1, 8))
        lanes = int(rng.integers(1, 4))
        rounds = int(rng.integers(-(-u // lanes), u + 1))
        w = [int(x) for x in rng.integers(0, 30, u)]
        rnd, lane, mk, exact = at.assign_grid(w, rounds, lanes, u_max=12)
        assert exact
        _valid(w, rnd, lane, rounds, lanes)
        assert mk == ref.makespan(w, lane, lanes)
        assert mk == ref.brute_force_makespan(w, rounds, lanes)


def test_greedy_bit_exact(augtree_lib):
    import shared_prompt_tree_gb300 as at
    rng = np.random.default_rng(8)
    for _ in range(100):
        u = int(rng.integers(1, 40))
        lanes = int(rng.integers(1, 9))
        rounds = int(rng.integers(-(-u // lanes), u + 1))
        w = [int(x) for x in rng.integers(0, 6, u)]  # many ties
        rnd, lane, mk, exact = at.assign_grid(w, rounds, lanes, u_max=0)
        assert not exact
        r_rnd, r_lane = ref.lpt(w, rounds, lanes)
        assert list(lane) == r_lane and list(rnd) == r_rnd
        assert mk == ref.makespan(w, r_lane, lanes)


def test_exact_never_worse_than_greedy(augtree_lib):
    import shared_prompt_tree_gb300 as at
    rng = np.random.default_rng(9)
    for _ in range(40):
        u = int(rng.integers(2, 13))
        lanes = int(rng.integers(2, 5))
        rounds = -(-u // lanes) + int(rng.integers(0, 2))
        w = [int(x) for x in rng.integers(1, 1000, u)]
        _, lane, mk, _ = at.assign_grid(w, rounds, lanes, u_max=12)
        _, _, mk_g, _ = at.assign_grid(w, rounds, lanes, u_max=0)
        assert mk <= mk_g
        assert mk >= max(max(w), -(-sum(w) // lanes))


def test_large_unit_count_falls_back_to_greedy(augtree_lib):
    import shared_prompt_tree_gb300 as at
    w = list(range(100, 0, -1))
    rnd, lane, mk, exact = at.assign_grid(w, 25, 4, u_max=16)
    assert not exact
    assert (list(rnd), list(lane)) == ref.lpt(w, 25, 4)


def test_invalid_arguments(augtree_lib):
    import shared_prompt_tree_gb300 as at
    for args in [([1, 2, 3], 1, 2, 12),    # 3 units, 2 cells
                 ([1, -2], 2, 2, 12),      # negative weight
                 ([1, 2], 0, 2, 12),       # no rounds
                 ([1, 2], 2, 0, 12),       # no lanes
                 ([1, 2], 2, 2, 17)]:      # cap above 16
        with pytest.raises(at.AugtreeError) as e:
            at.assign_grid(*args[:3], u_max=args[3])
        assert e.value.status == at.ERR_INVALID_ARG
    rnd, lane, mk, exact = at.assign_grid([], 1, 1)
    assert mk == 0 and len(rnd) == 0
