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


Item = Tuple[int, int, int, int, int, int]


def work_units(T: int, split: int = 1, tile_n: int = 256, num_kb: int = 1, sk_tiles: int = 0,
               sk_units: int = 0, tail_tiles: int = 0) -> List[List[Item]]:
    """The units the schedulers hand out, in unit order, each the list of its
    work items ``(record slot, grouped-order tile, first column, columns,
    first k-block, end k-block)``.

    * Whole tiles (``split == 1``, no stream-K region): unit u is tile u.
    * Column slices (``split`` 2 or 4): unit u is columns
      ``(u % split) * tile_n/split`` onwards of tile ``u // split``.
    * Tail halves (``tail_tiles = R > 0``, whole tiles otherwise): units
      ``0 .. T-R-1`` are those tiles, whole; then each of the last R tiles
      comes as two units, its left and then its right half of the columns.
    * Stream-K share (``sk_units = U > 0``): the first ``sk_tiles`` tiles form
      a region of ``L = sk_tiles * num_kb`` k-blocks, tile after tile.  Unit
      ``c < U`` owns the k-blocks ``x`` with ``floor(c*L/U) <= x <
      floor((c+1)*L/U)``; it has one item per tile those k-blocks fall in
      (record slot ``3c + j`` for its j-th such tile) and runs them last tile
      first.  Units ``U, U+1, ...`` are the remaining tiles, whole (record
      slots ``3U, 3U+1, ...``).  Items are listed in the order a unit runs
      them.

    The pages hand out whole tiles only; the column slices, the tail halves
    and the stream-K share are the library's additions for the tail of a
    grid (they change
    which cluster computes what, never the result beyond fp32 summation
    order).  The stream-K partition is written out here k-block by k-block,
    not by the closed forms the kernel uses, so the two can be compared.
    """
    if split not in (1, 2, 4) or (split > 1 and sk_units) or tail_tiles < 0 \
            or (tail_tiles and (split > 1 or sk_units or tail_tiles > T)):
        raise ValueError((split, sk_units, tail_tiles))
    units: List[List[Item]] = []
    if sk_units:
        U, L = sk_units, sk_tiles * num_kb
        if not (0 < sk_tiles <= T and U <= L):
            raise ValueError((T, sk_tiles, U, num_kb))
        starts = [c * L // U for c in range(U)]
        owner = []
        for x in range(L):
            c = 0
            while c + 1 < U and starts[c + 1] <= x:
                c += 1
            owner.append(c)
        for c in range(U):
            mine = [x for x in range(L) if owner[x] == c]
            items = []
            for j, t in enumerate(sorted({x // num_kb for x in mine})):
                ks = [x - t * num_kb for x in mine if x // num_kb == t]
                items.append((3 * c + j, t, 0, tile_n, min(ks), max(ks) + 1))
            units.append(items[::-1])
        for j in range(T - sk_tiles):
            units.append([(3 * U + j, sk_tiles + j, 0, tile_n, 0, num_kb)])
    elif split > 1:
        step = tile_n // split
        for u in range(T * split):
            units.append([(u, u // split, (u % split) * step, step, 0, num_kb)])
    else:
        for u in range(T - tail_tiles):
            units.append([(u, u, 0, tile_n, 0, num_kb)])
        half = tile_n // 2
        for t in range(T - tail_tiles, T):
            for h in (0, 1):
                units.append([(len(units), t, h * half, half, 0, num_kb)])
    return units


def work_items(T: int, split: int = 1, tile_n: int = 256, num_kb: int = 1, sk_tiles: int = 0,
               sk_units: int = 0, tail_tiles: int = 0) -> List[Item]:
    """Every work item of :func:`work_units`, in unit order."""
    return [it for u in work_units(T, split, tile_n, num_kb, sk_tiles, sk_units, tail_tiles) for it in u]


def record_slots(T: int, split: int = 1, sk_tiles: int = 0, sk_units: int = 0, tail_tiles: int = 0) -> int:
    """Record slots of a launch: three per stream-K unit plus one per other unit."""
    if sk_units:
        return 3 * sk_units + T - sk_tiles
    return T * split + tail_tiles


def grouped_items(problems, BM: int, BN: int, group_m: int, kb=None) -> List[Tuple[int, int, int]]:
    """Work ids of a grouped launch (several independent GEMMs, one list of
    tiles): ``(problem, tile-row, tile-col)`` per work id, problem by problem,
    each problem's tiles in grouped order; a problem with M or N = 0 has no
    tiles.  ``problems``: sequence of (M, N).  With ``kb`` (k-blocks per tile
    of each problem) the problems are listed most k-blocks first, equal
    counts in the given order (longest processing time first); without it,
    in the given order."""
    order = list(range(len(problems)))
    if kb is not None:
        order.sort(key=lambda g: -kb[g])   # list.sort is stable
    out = []
    for g in order:
        M, N = problems[g]
        if M == 0 or N == 0:
            continue
        Tm, Tn = tile_grid(M, N, BM, BN)
        for w in range(Tm * Tn):
            tm, tn = swizzle(w, Tm, Tn, group_m)
            out.append((g, tm, tn))
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
