"""Pins for the tile-coverage model and the raster map (no GPU)."""
import itertools
import json
import math
import os
import random

import numpy as np
import pytest

from oracle import coverage as cv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tail_example.json")


def test_worked_tail_example_static_6t():
    g = json.load(open(GOLDEN))
    st = g["static"]
    s = cv.simulate(g["n_tiles"], cv.STATIC, resident=st["resident"], n_workers=st["planned_workers"])
    cv.check_schedule(s)
    assert s.makespan == st["makespan_t"]
    assert {str(w): seq for w, seq in s.sequences.items()} == st["sequences"]


def test_worked_tail_example_clc_4t():
    g = json.load(open(GOLDEN))
    c = g["clc"]
    for prefetch in (False, True):
        s = cv.simulate(g["n_tiles"], cv.CLC, resident=c["resident"], prefetch=prefetch)
        cv.check_schedule(s)
        assert s.makespan == c["makespan_t"]
        assert sorted(len(v) for v in s.sequences.values()) == [c["tiles_per_worker"]] * c["resident"]


def test_nonpersistent_also_balances_the_example():
    # The page notes the plain non-persistent grid also spreads the 12 blocks dynamically.
    s = cv.simulate(12, cv.NONPERSISTENT, resident=3)
    cv.check_schedule(s)
    assert s.makespan == 4
    assert s.owner == list(range(12))


@pytest.mark.parametrize("T", [1, 2, 5, 12, 147, 148, 149, 296, 297])
@pytest.mark.parametrize("R", [1, 3, 148])
def test_unit_cost_closed_forms(T, R):
    clc = cv.simulate(T, cv.CLC, resident=R)
    cv.check_schedule(clc)
    assert clc.makespan == math.ceil(T / R)
    npers = cv.simulate(T, cv.NONPERSISTENT, resident=R)
    assert npers.makespan == math.ceil(T / R)
    W = 148
    st = cv.simulate(T, cv.STATIC, resident=R, n_workers=W)
    cv.check_schedule(st)
    per_worker = math.ceil(T / W)
    busy = min(W, T)
    # workers run in waves of R slots, each wave as long as its longest worker
    waves = math.ceil(busy / R)
    if busy <= R:
        assert st.makespan == per_worker
    else:
        assert per_worker <= st.makespan <= waves * per_worker
    assert st.owner == cv.expected_owner_static(T, W)


def test_static_planned_above_resident_tail():
    # 74 planned clusters on 62 resident, 4096 unit tiles: workers 0..25 own 56 tiles,
    # 26..73 own 55.  The 55-tile workers among the first 62 free their slots at 55,
    # and the 12 late workers (55 tiles each) then run to 110.
    st = cv.simulate(4096, cv.STATIC, resident=62, n_workers=74)
    assert st.makespan == 110
    clc = cv.simulate(4096, cv.CLC, resident=62)
    assert clc.makespan == math.ceil(4096 / 62)


def _check_every_order_once(schedules, T, R):
    """With the plain fetch (a worker cancels when its tile ends) the R first launches start
    at once and each later launch is obtained by exactly one successful cancel, one at a
    time, each choosing freely among the launches still pending ("CUTLASS CLC dynamic
    persistent kernel", section "What is cancelled is a launch, what is obtained is a work
    coordinate": only atomicity is fixed).  The orders in which launches R .. T-1 are
    cancelled are therefore exactly the permutations of those ids, (T - R)! of them, and an
    exhaustive enumeration must produce each once."""
    seqs = [tuple(s.cancelled) for s in schedules]
    expected = set(itertools.permutations(range(R, T)))
    assert len(seqs) == math.factorial(max(T - R, 0)), "number of cancel orders"
    assert len(set(seqs)) == len(seqs), "an order was enumerated twice"
    assert set(seqs) == expected, "the enumerated orders are not the permutations of the pending launches"


@pytest.mark.parametrize("T,R", [(1, 1), (2, 1), (4, 1), (6, 1), (3, 2), (5, 2), (6, 3), (7, 3), (7, 2), (2, 5)])
def test_cancel_orders_are_all_permutations_once(T, R):
    scheds = list(cv.enumerate_clc_orders(T, R))
    for s in scheds:
        cv.check_schedule(s)
    _check_every_order_once(scheds, T, R)
    if R == 1:
        # one resident worker: launch 0 runs its own tile, then the cancelled ones in order
        for s in scheds:
            assert s.sequences == {0: [0] + list(s.cancelled)}
            assert s.makespan == T


def test_truncated_or_repeating_enumerations_are_caught():
    """Planted mistakes in an enumerator: stopping after the first branch, or yielding a
    schedule twice, must fail the check above."""
    T, R = 5, 2
    with pytest.raises(AssertionError):
        _check_every_order_once(itertools.islice(cv.enumerate_clc_orders(T, R), 1), T, R)
    scheds = list(cv.enumerate_clc_orders(T, R))
    with pytest.raises(AssertionError):
        _check_every_order_once(scheds[:-1] + scheds[:1], T, R)
    with pytest.raises(AssertionError):
        _check_every_order_once(scheds[:-1], T, R)


def _brute_force_choice_sequences(T, R, prefetch, cost):
    """Every sequence of choices the model can make, found without the enumerator's search:
    run the model once for every tuple of T choice indices (index i picks the i-th smallest
    pending launch) and keep the tuples whose every used index was valid; the used prefix
    of such a tuple is one distinct schedule."""
    found = set()
    for idx in itertools.product(range(max(T, 1)), repeat=T):
        used = []
        bad = []

        def pick(pending):
            k = idx[len(used)]
            used.append(k)
            if k >= len(pending):
                bad.append(k)
                return sorted(pending)[0]
            return sorted(pending)[k]

        cv.simulate(T, cv.CLC, R, cost=cost, pick=pick, prefetch=prefetch)
        if not bad:
            found.add(tuple(used))
    return found


@pytest.mark.parametrize("T,R", [(1, 1), (3, 1), (3, 2), (4, 2), (5, 2), (5, 3)])
@pytest.mark.parametrize("prefetch", [False, True])
def test_enumeration_matches_brute_force(T, R, prefetch):
    """The enumerator's schedules are exactly the model's reachable choice sequences, each
    once (also with the overlapped fetch, where no closed form counts them)."""
    rng = random.Random(T * 10 + R)
    cost = [rng.choice([0.5, 1.0, 2.0]) for _ in range(T)]
    got = []
    for s in cv.enumerate_clc_orders(T, R, prefetch=prefetch, cost=cost):
        cv.check_schedule(s)
        got.append(tuple(s.cancelled))
    # map each brute-force choice sequence to its cancelled-launch sequence
    expected = set()
    for choices in _brute_force_choice_sequences(T, R, prefetch, cost):
        it = iter(choices)
        s = cv.simulate(T, cv.CLC, R, cost=cost, pick=lambda p: sorted(p)[next(it)], prefetch=prefetch)
        expected.add(tuple(s.cancelled))
    assert len(got) == len(set(got)) == len(expected)
    assert set(got) == expected


def test_exhaustive_with_uneven_costs():
    rng = random.Random(5)
    for _ in range(20):
        T = rng.randint(1, 6)
        R = rng.randint(1, 3)
        cost = [rng.choice([0.5, 1.0, 2.0, 3.0]) for _ in range(T)]
        for s in cv.enumerate_clc_orders(T, R, cost=cost):
            cv.check_schedule(s)
            assert s.makespan >= max(cost)


def test_planted_double_claim_is_caught():
    s = cv.simulate(6, cv.CLC, resident=2)
    s.claims[3] = 2
    with pytest.raises(AssertionError):
        cv.check_schedule(s)


@pytest.mark.parametrize("mt,nt,G", [(1, 1, 8), (3, 4, 8), (24, 32, 8), (17, 5, 8), (5, 7, 1), (9, 3, 4), (64, 32, 8)])
def test_raster_is_a_bijection(mt, nt, G):
    seen = {cv.raster(c, mt, nt, G) for c in range(mt * nt)}
    assert seen == {(m, n) for m in range(mt) for n in range(nt)}


def test_raster_closed_forms():
    mt, nt = 6, 5
    # one band covering all rows: column-major order
    assert [cv.raster(c, mt, nt, 8) for c in range(mt * nt)] == [(c % mt, c // mt) for c in range(mt * nt)]
    # band height 1: row-major order
    assert [cv.raster(c, mt, nt, 1) for c in range(mt * nt)] == [(c // nt, c % nt) for c in range(mt * nt)]
    # 17 rows in bands of 8: the last band has one row, walked along n
    assert [cv.raster(16 * 5 + j, 17, 5, 8) for j in range(5)] == [(16, j) for j in range(5)]
    assert cv.raster(1, 17, 5, 8) == (1, 0) and cv.raster(8, 17, 5, 8) == (0, 1)


def test_grouped_tile_offsets():
    tiles_m = [1, 3, 2]
    nt = 2
    out = [cv.grouped_tile(c, tiles_m, nt) for c in range(12)]
    assert out[0] == (0, 0, 0) and out[1] == (0, 0, 1)
    assert out[2] == (1, 0, 0) and out[3] == (1, 1, 0) and out[5] == (1, 0, 1)
    assert out[8] == (2, 0, 0) and out[11] == (2, 1, 1)
    with pytest.raises(ValueError):
        cv.grouped_tile(12, tiles_m, nt)


def test_device_log_checker_accepts_and_rejects():
    T, W = 10, 4
    owner = cv.expected_owner_static(T, W)
    cv.check_device_log(cv.STATIC, owner, [1] * T, [0, 1, 2, 3], W, n_workers=W)
    with pytest.raises(AssertionError):
        cv.check_device_log(cv.STATIC, owner, [1] * 9 + [0], [0, 1, 2, 3], W, n_workers=W)
    # CLC: launches 0..2 ran, 3..5 were stolen
    owner = [0, 1, 2, 0, 1, 2]
    first = [0, 1, 2, -1, -1, -1]
    cv.check_device_log(cv.CLC, owner, [1] * 6, first, 6)
    with pytest.raises(AssertionError):   # launch 3 ran although tile 3 was stolen by 0
        cv.check_device_log(cv.CLC, [0, 1, 2, 0, 3, 2], [1] * 6, [0, 1, 2, 3, -1, -1], 6)
    with pytest.raises(AssertionError):   # a worker did not start with its own tile
        cv.check_device_log(cv.CLC, owner, [1] * 6, [0, 1, 3, -1, -1, -1], 6)


def test_grouped_tile_per_problem_columns():
    tiles_m, nts = [2, 1, 3], [1, 3, 2]
    out = [cv.grouped_tile(c, tiles_m, nts) for c in range(2 + 3 + 6)]
    assert out[:2] == [(0, 0, 0), (0, 1, 0)]
    assert out[2:5] == [(1, 0, 0), (1, 0, 1), (1, 0, 2)]
    assert out[5:] == [(2, 0, 0), (2, 1, 0), (2, 2, 0), (2, 0, 1), (2, 1, 1), (2, 2, 1)]
    # the same as the uniform form when every problem has the same column count
    assert [cv.grouped_tile(c, [2, 3], [4, 4]) for c in range(20)] == [cv.grouped_tile(c, [2, 3], 4) for c in range(20)]


def test_greedy_schedules_respect_the_list_scheduling_bound():
    """CLC (fetch when a tile ends) and non-persistent launches never leave a slot idle while
    a tile is pending, so they are greedy list schedules: for tile costs c on R slots the
    makespan lies between sum(c)/R and sum(c)/R + (1 - 1/R) max(c) (Graham's bound for list
    scheduling).  Static scheduling is not greedy and may exceed it."""
    rng = np.random.default_rng(17)
    exceeded = 0
    for _ in range(300):
        T = int(rng.integers(1, 60))
        R = int(rng.integers(1, 12))
        cost = list(rng.uniform(0.1, 5.0, size=T))
        lo, hi = sum(cost) / R, sum(cost) / R + (1 - 1 / R) * max(cost)
        for mode in (cv.CLC, cv.NONPERSISTENT):
            s = cv.simulate(T, mode, R, cost=cost)
            cv.check_schedule(s)
            assert lo - 1e-9 <= s.makespan <= hi + 1e-9, (mode, T, R, s.makespan, lo, hi)
        st = cv.simulate(T, cv.STATIC, R, n_workers=R + int(rng.integers(0, 3)), cost=cost)
        cv.check_schedule(st)
        exceeded += st.makespan > hi + 1e-9
    assert exceeded > 0, "static should exceed the greedy bound on some uneven draws"
