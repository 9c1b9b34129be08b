"""What the three tile schedulers compute (test infrastructure).

Only tests, smoke() and bench.py's CPU legs use this module; it never imports
the CUDA package.

Sources ("Persistent Kernels with Cluster Launch Control", first two
paragraphs and "Choosing between static and CLC scheduling"; "question about
persistent kernel concept", the question):

* The output is cut into ``T = Tm * Tn`` tiles.  A linear work id ``w`` in
  ``[0, T)`` is mapped to a tile ``(tm, tn)`` by the GROUP_SIZE_M grouped
  ordering named in "[Persistent] Performance on 09-persistent-matmul on A100
  worse than non-persistent" (its hyperparameter list).  The pages name the
  parameter but not the formula; the reading used is the usual grouped order:
  work ids walk down a group of at most GROUP_SIZE_M tile-rows column by
  column, the last group being shorter.
* non-persistent: one cluster per tile; cluster ``c`` does work id ``c``.
* static persistent: ``G`` resident clusters; cluster ``c`` does
  ``c, c + G, c + 2G, ...`` (later tiles derived in software, deterministic).
* CLC persistent: the grid has one cluster per tile.  A running cluster first
  does its own id, then asks the hardware to cancel a cluster that has not
  launched yet and does that cluster's id.  After one failed request it must
  not ask again.  Every tile is done exactly once: either its own cluster
  launched and did it, or the cluster that cancelled it did.
"""
from __future__ import annotations

import random
from typing import Dict, List, Optional, Tuple


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def tile_grid(M: int, N: int, BM: int, BN: int) -> Tuple[int, int]:
    """Number of tile-rows and tile-columns covering an M x N output."""
    return cdiv(M, BM), cdiv(N, BN)


def swizzle(w: int, Tm: int, Tn: int, group_m: int) -> Tuple[int, int]:
    """Work id -> (tile-row, tile-col) in GROUP_SIZE_M grouped order."""
    if not 0 <= w < Tm * Tn:
        raise IndexError(w)
    per_group = group_m * Tn
    group = w // per_group
    first_m = group * group_m
    rows_here = min(Tm - first_m, group_m)
    r = w - group * per_group
    return first_m + r % rows_here, r // rows_here


def work_items(T: int, full_work: int, split: int, tile_n: int = 256, split_k: bool = False,
               num_kb: int = 1, part_kb: Optional[int] = None) -> List[Tuple[int, int, int, int, int, int]]:
    """(work id, grouped-order tile index, first column, columns, first k-block,
    end k-block) of every work item.

    Work ids below ``full_work`` are whole tiles.  Each remaining tile is cut
    into ``split`` parts: work id ``full_work + split*j + h`` is part h of
    tile ``full_work + j``.  Parts are column slices of ``tile_n / split``
    columns, or (``split_k``) k-block ranges whose partial sums add up to the
    tile: parts 0..split-2 take ``part_kb`` k-blocks each (default
    ``num_kb // split``), part h covering ``[h*part_kb, (h+1)*part_kb)``, and
    the last part takes the rest, up to ``num_kb``.  Cutting
    tiles changes how the output is partitioned among CTAs, never what is
    computed ("Neither mode creates additional independent work at the tail
    of a grid": cutting is a separate device for the last wave).
    """
    if not (0 <= full_work <= T and 1 <= split <= 4):
        raise ValueError((T, full_work, split))
    if not split_k and split not in (1, 2, 4):
        raise ValueError(split)
    a = (num_kb // split) if part_kb is None else part_kb
    if split_k and not (1 <= a and (split - 1) * a < num_kb):
        raise ValueError((num_kb, split, a))
    out = [(w, w, 0, tile_n, 0, num_kb) for w in range(full_work)]
    for j in range(T - full_work):
        for h in range(split):
            w = full_work + split * j + h
            if split_k:
                out.append((w, full_work + j, 0, tile_n, h * a, num_kb if h == split - 1 else (h + 1) * a))
            else:
                step = tile_n // split
                out.append((w, full_work + j, h * step, step, 0, num_kb))
    return out


def static_grid(T: int, max_clusters: int) -> int:
    """Resident clusters launched by the static persistent scheduler."""
    return max(1, min(T, max_clusters)) if T > 0 else 0


def static_assignment(T: int, G: int) -> List[Tuple[int, int, int]]:
    """(work id, cluster, iteration) for every tile the static scheduler runs.

    Cluster c walks its own sequence c, c + G, ... until it leaves [0, T)."""
    out = []
    for c in range(G):
        w, it = c, 0
        while w < T:
            out.append((w, c, it))
            w, it = w + G, it + 1
    return out


def nonpersistent_assignment(T: int) -> List[Tuple[int, int, int]]:
    """(work id, cluster, iteration) when every cluster does one tile."""
    return [(c, c, 0) for c in range(T)]


def clc_replay(T: int, resident: int, cost=None, fail_at: Optional[Dict[int, int]] = None,
               seed: int = 0):
    """Event replay of CLC work stealing on ``resident`` cluster slots.

    Clusters launch in id order whenever a slot is free.  A running cluster
    finishes its current tile after ``cost(w)`` time units, then issues one
    ``try_cancel``: it succeeds with the lowest not-yet-launched cluster id
    (the order the hardware picks is not stated; this is one admissible
    choice), and fails when every cluster has launched or been cancelled.
    ``fail_at[c] = n`` forces the n-th request of cluster c to fail (an
    injected failure).  After a failure the cluster stops and never asks
    again.

    Returns (list of (work id, cluster, iteration), requests per cluster,
    requests issued after a failure).
    """
    rng = random.Random(seed)
    cost = cost or (lambda w: 1.0 + rng.random())
    fail_at = fail_at or {}
    next_launch = 0          # lowest cluster id neither launched nor cancelled
    events: List[Tuple[int, int, int]] = []
    requests: Dict[int, int] = {}
    after_fail = 0
    running: List[Tuple[float, int, int, int]] = []   # (finish time, cluster, work id, iter)
    failed = set()
    now = 0.0

    def launch_one(t0: float) -> bool:
        nonlocal next_launch
        if next_launch >= T:
            return False
        c = next_launch
        next_launch += 1
        events.append((c, c, 0))
        running.append((t0 + cost(c), c, c, 0))
        return True

    while len(running) < resident and launch_one(now):
        pass
    while running:
        running.sort()
        now, c, w, it = running.pop(0)
        n = requests.get(c, 0)
        if c in failed:
            after_fail += 1
        requests[c] = n + 1
        forced = fail_at.get(c) == n
        if not forced and next_launch < T:
            victim = next_launch
            next_launch += 1
            events.append((victim, c, it + 1))
            running.append((now + cost(victim), c, victim, it + 1))
        else:
            failed.add(c)
            while len(running) < resident and launch_one(now):
                pass
    return events, requests, after_fail


def coverage(events: List[Tuple[int, int, int]], T: int) -> List[int]:
    """Visit count per work id (every entry must be exactly 1)."""
    visits = [0] * T
    for w, _, _ in events:
        visits[w] += 1
    return visits
