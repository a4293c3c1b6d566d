"""Tile-coverage model of the three scheduling policies (TEST INFRASTRUCTURE ONLY).

Only the tests, the package smoke check and the benchmark's CPU baseline import this
module.  It shares no code with the CUDA path.

What it models ("CUTLASS CLC dynamic persistent kernel"):

* Section "From one tile per block to one worker working continuously", table:
  - non-persistent: the grid is launched over all tiles; each block computes its own
    tile and exits;
  - static persistent: the grid is launched over a preset number of workers, and each
    worker walks a sequence fixed in advance;
  - CLC dynamic persistent: the grid is launched over all tiles; a running worker takes
    over launches that have not started yet.
* Section "Why a fixed task sequence has a tail": with 12 tiles, 4 planned workers at
  stride 4 and only 3 resident, the static makespan is about 6t; with CLC and 3
  concurrent workers each worker runs 4 tiles and the makespan is about 4t (a hand
  calculation, not a measurement).
* Section "What is cancelled is a launch, what is obtained is a work coordinate": the
  cancel is atomic, so a coordinate is never in two successful responses of one grid;
  every tile is computed either by its own launch or by exactly one stealing worker; a
  block that is already running cannot be taken over.  A worker's first tile is the
  one of its own launch coordinate (the ClcID), later tiles come from CLC.
* Section "Cluster granularity and exit after failure": a failed cancel only tells the
  worker to stop fetching; it never yields a coordinate.

Readings where the pages are silent (each listed in the design notes):
* which pending launch a successful cancel returns is not specified, so the model takes
  it as a free choice (``pick``); the default is the lowest pending launch id;
* the hardware starts pending launches in ascending id order when a slot frees;
* tile ids here are *linear* launch ids; ``raster`` maps them to output tiles.
"""
from __future__ import annotations

import heapq
import itertools
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence, Tuple

NONPERSISTENT = "nonpersistent"
STATIC = "static"
CLC = "clc"
MODES = (CLC, STATIC, NONPERSISTENT)


# --------------------------------------------------------------------------------------
# Raster / swizzle map (linear tile id -> output tile coordinate)
# --------------------------------------------------------------------------------------
def raster(c: int, mt: int, nt: int, group_rows: int = 8) -> Tuple[int, int]:
    """Map linear tile id ``c`` of an ``mt x nt`` tile grid to its tile (m, n).

    The pages name the swizzle / raster step applied after decoding a response (page
    "CUTLASS CLC dynamic persistent kernel", section "Following the CUTLASS source";
    CuTeDSL ``_swizzle_and_rasterize`` in the task-scheduling walk-through) without
    defining it.  Reading used here: tiles are taken in bands of ``group_rows`` tile
    rows; inside a band the row index runs fastest (column-major), and the last band
    may be shorter.  ``group_rows == 1`` is plain row-major order.
    """
    if not (0 <= c < mt * nt):
        raise ValueError(f"tile id {c} outside a {mt}x{nt} grid")
    if group_rows < 1:
        raise ValueError("group_rows must be >= 1")
    band = c // (group_rows * nt)
    rows_in_band = min(group_rows, mt - band * group_rows)
    r = c - band * group_rows * nt
    return band * group_rows + r % rows_in_band, r // rows_in_band


def grouped_tile(c: int, tiles_m: Sequence[int], nt, group_rows: int = 8) -> Tuple[int, int, int]:
    """Flat tile id over several problems -> (group, m, n).

    Problems are laid out one after another in the flat id (problem g owns the ids
    from sum_{h<g} tiles_m[h]*nt[h] on), and the same raster map applies inside each.
    ``nt`` is one tile-column count for all problems or one per problem.
    """
    nts = list(nt) if isinstance(nt, (list, tuple)) else [nt] * len(tiles_m)
    base = 0
    for g, (mt, ntg) in enumerate(zip(tiles_m, nts)):
        cnt = mt * ntg
        if c < base + cnt:
            m, n = raster(c - base, mt, ntg, group_rows)
            return g, m, n
        base += cnt
    raise ValueError(f"flat tile id {c} beyond {base} tiles")


# --------------------------------------------------------------------------------------
# Discrete-event model of the three policies
# --------------------------------------------------------------------------------------
@dataclass
class Schedule:
    mode: str
    n_tiles: int
    n_launch: int
    owner: List[int]                     # linear tile id -> launch id of the worker that ran it
    sequences: Dict[int, List[int]]      # worker (launch id that ran) -> tiles, in order
    cancelled: List[int]                 # launch ids whose launch was cancelled (CLC only)
    start: List[float]
    end: List[float]
    makespan: float
    claims: List[int] = field(default_factory=list)


Picker = Callable[[List[int]], int]


def lowest(pending: List[int]) -> int:
    return min(pending)


def simulate(n_tiles: int, mode: str, resident: int, n_workers: Optional[int] = None,
             cost: Optional[Sequence[float]] = None, pick: Picker = lowest,
             prefetch: bool = False) -> Schedule:
    """Run one schedule of ``n_tiles`` tiles on ``resident`` concurrent worker slots.

    mode        one of ``clc``, ``static``, ``nonpersistent``.
    n_workers   static only: the planned worker count W (worker w owns w, w+W, ...).
    cost        per-tile duration (default 1 each).
    pick        CLC: chooses which pending launch a successful cancel returns.
    prefetch    CLC: the next tile is claimed when the current one starts (the
                overlapped fetch) instead of when it ends (the pages' plain loop).
    """
    if mode not in MODES:
        raise ValueError(mode)
    if resident < 1:
        raise ValueError("need at least one resident slot")
    cost = [1.0] * n_tiles if cost is None else list(cost)
    if len(cost) != n_tiles:
        raise ValueError("cost length")

    if mode == STATIC:
        W = n_workers if n_workers is not None else resident
        if W < 1:
            raise ValueError("static needs >= 1 worker")
        plan = {w: list(range(w, n_tiles, W)) for w in range(W)}
        n_launch = W
    else:
        plan = {t: [t] for t in range(n_tiles)}
        n_launch = n_tiles

    owner = [-1] * n_tiles
    claims = [0] * n_tiles
    start = [0.0] * n_tiles
    end = [0.0] * n_tiles
    seqs: Dict[int, List[int]] = {}
    cancelled: List[int] = []
    pending = list(range(n_launch))          # launches the hardware has not started
    events: List[Tuple[float, int, int]] = []  # (time a worker becomes free, order, worker)
    order = itertools.count()
    state: Dict[int, dict] = {}

    def claim(w: int) -> Optional[int]:
        """CLC try_cancel by worker w: a pending launch's tile, or None on failure."""
        if not pending:
            return None
        v = pick(list(pending))
        if v not in pending:
            raise ValueError("picker returned a launch that is not pending")
        pending.remove(v)
        cancelled.append(v)
        return v

    def run_tile(w: int, t: int, now: float) -> float:
        owner[t] = w
        claims[t] += 1
        seqs.setdefault(w, []).append(t)
        start[t] = now
        end[t] = now + cost[t]
        return end[t]

    def launch(now: float) -> None:
        """A slot is free: the hardware starts the lowest pending launch."""
        while pending:
            w = pending.pop(0)
            st = {"queue": list(plan[w]), "next": None}
            state[w] = st
            if st["queue"]:
                break
            # a static worker with no tile (W > tiles) exits at once, freeing the slot
        else:
            return
        t = st["queue"].pop(0)            # own coordinate first
        finish = run_tile(w, t, now)
        if mode == CLC and prefetch:
            st["next"] = claim(w)
        heapq.heappush(events, (finish, next(order), w))

    for _ in range(min(resident, n_launch)):
        launch(0.0)

    makespan = 0.0
    while events:
        now, _, w = heapq.heappop(events)
        makespan = max(makespan, now)
        st = state[w]
        if mode == CLC:
            nxt = st["next"] if prefetch else claim(w)
            st["next"] = None
            if nxt is None:               # failed cancel: stop fetching, the worker exits
                launch(now)
                continue
            finish = run_tile(w, nxt, now)
            if prefetch:
                st["next"] = claim(w)
            heapq.heappush(events, (finish, next(order), w))
        else:
            if st["queue"]:
                finish = run_tile(w, st["queue"].pop(0), now)
                heapq.heappush(events, (finish, next(order), w))
            else:
                launch(now)

    return Schedule(mode, n_tiles, n_launch, owner, seqs, cancelled, start, end,
                    makespan, claims)


# --------------------------------------------------------------------------------------
# Invariants (the model's and the device log's)
# --------------------------------------------------------------------------------------
def check_schedule(s: Schedule) -> None:
    """Assert the coverage invariant on a model schedule."""
    assert all(c == 1 for c in s.claims), "a tile was not computed exactly once"
    assert sum(s.claims) == s.n_tiles
    workers = set(s.sequences)
    if s.mode == CLC:
        for w, seq in s.sequences.items():
            assert seq[0] == w, "a worker's first tile is its own launch coordinate"
        assert not (workers & set(s.cancelled)), "a cancelled launch never runs"
        assert len(workers) + len(s.cancelled) == s.n_launch
        assert len(set(s.cancelled)) == len(s.cancelled), "a launch cancelled twice"
    for t, w in enumerate(s.owner):
        if s.mode == CLC:
            assert (w == t) == (t not in s.cancelled)


def expected_owner_static(n_tiles: int, n_workers: int) -> List[int]:
    """Static persistent: linear tile t is run by worker t mod W."""
    return [t % n_workers for t in range(n_tiles)]


def expected_owner_nonpersistent(n_tiles: int) -> List[int]:
    """Non-persistent: linear tile t is run by launch t."""
    return list(range(n_tiles))


def check_device_log(mode: str, owner_lin: Sequence[int], claims_lin: Sequence[int],
                     first_of_worker: Sequence[int], n_launch: int,
                     n_workers: Optional[int] = None) -> None:
    """Check a device ownership log, re-indexed by linear tile id, against the model.

    owner_lin[t]   worker (launch id) that computed linear tile t
    claims_lin[t]  how many times tile t was computed
    first_of_worker[w]  first linear tile worker w computed, or -1 if it never ran
    """
    T = len(owner_lin)
    bad = [t for t in range(T) if claims_lin[t] != 1]
    assert not bad, f"tiles not claimed exactly once: {bad[:10]}"
    assert sum(claims_lin) == T
    if mode == STATIC:
        exp = expected_owner_static(T, n_workers)
        assert list(owner_lin) == exp, "static owner map differs from t mod W"
        for w in range(n_workers):
            assert first_of_worker[w] == (w if w < T else -1)
    elif mode == NONPERSISTENT:
        assert list(owner_lin) == expected_owner_nonpersistent(T)
        assert list(first_of_worker[:T]) == list(range(T))
    else:
        ran = {w for w in range(n_launch) if first_of_worker[w] != -1}
        for w in ran:
            assert first_of_worker[w] == w, f"worker {w} did not start with its own tile"
        assert set(owner_lin) == ran, "a worker id in the log never ran, or a runner has no tile"
        for t in range(T):
            stolen = owner_lin[t] != t
            assert stolen == (t not in ran), f"tile {t}: own launch ran but tile was stolen, or vice versa"


def enumerate_clc_orders(n_tiles: int, resident: int, prefetch: bool = False,
                         cost: Optional[Sequence[float]] = None):
    """Yield every CLC schedule over all choices of which pending launch each
    successful cancel returns (the pages fix only atomicity, not the order)."""
    def run(prefix: List[int]):
        choices: List[int] = []
        branch_sizes: List[int] = []

        def pick(pending: List[int]) -> int:
            i = len(choices)
            k = prefix[i] if i < len(prefix) else 0
            branch_sizes.append(len(pending))
            choices.append(k)
            return sorted(pending)[k]

        s = simulate(n_tiles, CLC, resident, cost=cost, pick=pick, prefetch=prefetch)
        return s, choices, branch_sizes

    stack = [[]]
    while stack:
        prefix = stack.pop()
        s, choices, sizes = run(prefix)
        yield s
        for i in range(len(prefix), len(choices)):
            for alt in range(1, sizes[i]):
                stack.append(choices[:i] + [alt])
