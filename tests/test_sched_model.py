"""Pins for the scheduler model (host logic, no GPU).

The model states what each scheduler must do; these tests check it against
hand-worked orders, closed forms of the grouped order at its extremes, and the
coverage invariant: neither scheduler adds or drops work ("Choosing between
static and CLC scheduling"), so every tile is done exactly once.
"""
import json
import os
import random

import pytest

from oracle import sched as sm

# (M, N, BM, BN) for every workload and both tile shapes (128x256 per CTA,
# 256x256 per CTA pair)
GRIDS = sorted({
    (m, n, bm, bn)
    for (m, n) in [(512, 512), (4096, 4096), (8192, 8192), (5120, 5120), (4224, 3968),
                   (19200, 256), (1, 1), (129, 257)]
    for (bm, bn) in [(128, 256), (256, 256)]
})


def test_swizzle_hand_worked(golden_dir):
    with open(os.path.join(golden_dir, "swizzle_3x2_g2.json")) as f:
        g = json.load(f)
    got = [list(sm.swizzle(w, g["Tm"], g["Tn"], g["group_m"])) for w in range(g["Tm"] * g["Tn"])]
    assert got == g["order"]


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("group_m", [1, 8])
def test_swizzle_is_a_bijection(grid, group_m):
    Tm, Tn = sm.tile_grid(*grid)
    seen = {sm.swizzle(w, Tm, Tn, group_m) for w in range(Tm * Tn)}
    assert seen == {(i, j) for i in range(Tm) for j in range(Tn)}


def test_swizzle_extremes():
    Tm, Tn = 5, 7
    # one row per group: plain row-major order
    assert [sm.swizzle(w, Tm, Tn, 1) for w in range(Tm * Tn)] == \
        [(w // Tn, w % Tn) for w in range(Tm * Tn)]
    # a group taller than the grid: plain column-major order
    assert [sm.swizzle(w, Tm, Tn, 8) for w in range(Tm * Tn)] == \
        [(w % Tm, w // Tm) for w in range(Tm * Tn)]


def test_tile_counts_of_the_workloads():
    assert sm.tile_grid(512, 512, 128, 256) == (4, 2)
    assert sm.tile_grid(4096, 4096, 128, 256) == (32, 16)
    assert sm.tile_grid(5120, 5120, 128, 256) == (40, 20)
    assert sm.tile_grid(4224, 3968, 128, 256) == (33, 16)       # 528 tiles
    assert sm.tile_grid(19200, 256, 128, 256) == (150, 1)


@pytest.mark.parametrize("T,G", [(8, 148), (512, 148), (2048, 148), (150, 148), (1, 1), (528, 74)])
def test_static_covers_exactly_once(T, G):
    G = sm.static_grid(T, G)
    ev = sm.static_assignment(T, G)
    assert sm.coverage(ev, T) == [1] * T
    per = {}
    for _, c, _ in ev:
        per[c] = per.get(c, 0) + 1
    assert max(per.values()) - min(per.values()) <= 1      # balanced to one tile
    for w, c, it in ev:
        assert c == w % G and it == w // G


def test_nonpersistent_is_identity():
    ev = sm.nonpersistent_assignment(37)
    assert sm.coverage(ev, 37) == [1] * 37
    assert all(w == c and it == 0 for w, c, it in ev)


@pytest.mark.parametrize("T,resident", [(1, 148), (8, 148), (150, 148), (512, 148), (2048, 148),
                                        (1024, 74), (800, 10)])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_clc_replay_covers_exactly_once(T, resident, seed):
    ev, req, after_fail = sm.clc_replay(T, resident, seed=seed)
    assert sm.coverage(ev, T) == [1] * T
    assert after_fail == 0
    # a cluster's first tile is its own id
    firsts = {(c, w) for w, c, it in ev if it == 0}
    assert all(c == w for c, w in firsts)


@pytest.mark.parametrize("seed", range(5))
def test_clc_replay_with_injected_failures(seed):
    rnd = random.Random(seed)
    T, resident = 600, 40
    fail_at = {c: rnd.randrange(0, 4) for c in rnd.sample(range(T), 60)}
    ev, req, after_fail = sm.clc_replay(T, resident, fail_at=fail_at, seed=seed)
    assert sm.coverage(ev, T) == [1] * T        # un-cancelled clusters run their own tile
    assert after_fail == 0


def test_clc_replay_uneven_costs_cover_exactly_once():
    # tile costs that differ by 5x change who runs what, never how often
    T, resident = 200, 20
    ev, _, _ = sm.clc_replay(T, resident, cost=lambda w: 5.0 if w % 2 == 0 else 1.0)
    assert sm.coverage(ev, T) == [1] * T


def test_work_items_hand_worked():
    # whole tiles; a sub-wave problem cut into column slices of 128 and 64 columns
    assert sm.work_items(3, num_kb=8) == [(0, 0, 0, 256, 0, 8), (1, 1, 0, 256, 0, 8), (2, 2, 0, 256, 0, 8)]
    assert sm.work_items(2, 2, num_kb=8) == [
        (0, 0, 0, 128, 0, 8), (1, 0, 128, 128, 0, 8), (2, 1, 0, 128, 0, 8), (3, 1, 128, 128, 0, 8)]
    assert [i[2:4] for i in sm.work_items(2, 4)[:4]] == [(0, 64), (64, 64), (128, 64), (192, 64)]
    with pytest.raises(ValueError):
        sm.work_items(4, 3)
    with pytest.raises(ValueError):      # slices and the stream-K share exclude each other
        sm.work_items(4, 2, num_kb=4, sk_tiles=4, sk_units=2)


def test_stream_k_hand_worked(golden_dir):
    with open(os.path.join(golden_dir, "stream_k_T5_G3_kb4.json")) as f:
        g = json.load(f)
    units = sm.work_units(g["T"], num_kb=g["num_kb"], sk_tiles=g["sk_tiles"], sk_units=g["sk_units"])
    assert [[list(it) for it in u] for u in units] == g["units"]
    assert sm.record_slots(g["T"], sk_tiles=g["sk_tiles"], sk_units=g["sk_units"]) == g["slots"]
    pieces = {}
    for it in sm.work_items(g["T"], num_kb=g["num_kb"], sk_tiles=g["sk_tiles"], sk_units=g["sk_units"]):
        pieces[it[1]] = pieces.get(it[1], 0) + 1
    assert sorted(t for t, n in pieces.items() if n > 1) == g["cut_tiles"]
    # with whole tiles after the region: T = 8 on G = 3 -> R = 2, region = 5 tiles, 3 whole tiles
    units = sm.work_units(8, num_kb=4, sk_tiles=5, sk_units=3)
    assert units[:3] == sm.work_units(5, num_kb=4, sk_tiles=5, sk_units=3)
    assert units[3:] == [[(9, 5, 0, 256, 0, 4)], [(10, 6, 0, 256, 0, 4)], [(11, 7, 0, 256, 0, 4)]]


def test_tail_halves_hand_worked():
    # T = 5 with the last 2 tiles in column halves: 3 whole units, then 4 halves
    assert sm.work_units(5, num_kb=6, tail_tiles=2) == [
        [(0, 0, 0, 256, 0, 6)], [(1, 1, 0, 256, 0, 6)], [(2, 2, 0, 256, 0, 6)],
        [(3, 3, 0, 128, 0, 6)], [(4, 3, 128, 128, 0, 6)], [(5, 4, 0, 128, 0, 6)], [(6, 4, 128, 128, 0, 6)]]
    assert sm.record_slots(5, tail_tiles=2) == 7
    for bad in (dict(split=2, tail_tiles=1), dict(sk_tiles=4, sk_units=2, tail_tiles=1), dict(tail_tiles=6),
                dict(tail_tiles=-1)):
        with pytest.raises(ValueError):
            sm.work_units(5, num_kb=4, **bad)


@pytest.mark.parametrize("T,G", [(256, 76), (512, 152), (1024, 76), (320, 76), (4, 3), (41, 20), (21, 20)])
def test_tail_halves_partition_and_last_wave(T, G):
    """The last R = T mod G tiles in halves (when 2R <= G): every tile is still
    covered exactly once, and under the static assignment no cluster has more
    than half a tile in the last wave."""
    R = T % G
    assert 0 < 2 * R <= G
    units = sm.work_units(T, num_kb=3, tail_tiles=R)
    items = [it for u in units for it in u]
    assert [i[0] for i in items] == list(range(sm.record_slots(T, tail_tiles=R)))
    _cells_partition(items, T, 3)
    load = [0] * G                                       # in half tiles
    for u, its in enumerate(units):
        load[u % G] += sum(it[3] for it in its) // 128
    assert max(load) == 2 * (T // G) + 1 and min(load) == 2 * (T // G)


def _cells_partition(items, T, num_kb, tile_n=256):
    cells = {}
    for _, t, off, n, k0, k1 in items:
        assert k1 > k0
        cells.setdefault(t, set())
        new = {(c, kb) for c in range(off, off + n, 64) for kb in range(k0, k1)}
        assert not (cells[t] & new)                     # nothing computed twice
        cells[t] |= new
    assert sorted(cells) == list(range(T))
    for t in range(T):
        assert cells[t] == {(c, kb) for c in range(0, tile_n, 64) for kb in range(num_kb)}


@pytest.mark.parametrize("T,s", [(8, 4), (20, 2), (150, 1), (1, 4), (37, 2)])
def test_slices_partition_every_tile(T, s):
    items = sm.work_items(T, s, num_kb=3)
    assert [i[0] for i in items] == list(range(sm.record_slots(T, s)))
    _cells_partition(items, T, 3)


@pytest.mark.parametrize("T,G,num_kb", [(5, 3, 4), (8, 3, 4), (20, 7, 2), (20, 7, 9), (512, 152, 64),
                                        (256, 76, 64), (528, 152, 32), (800, 152, 1), (153, 152, 3),
                                        (303, 152, 5), (1024, 76, 128), (11, 10, 1), (19, 10, 7)])
def test_stream_k_partition_and_balance(T, G, num_kb):
    R = T % G
    sk_tiles = R + G
    units = sm.work_units(T, num_kb=num_kb, sk_tiles=sk_tiles, sk_units=G)
    items = [it for u in units for it in u]
    assert len(units) == G + T - sk_tiles
    _cells_partition(items, T, num_kb)
    slots = [it[0] for it in items]
    assert len(set(slots)) == len(slots) and max(slots) < sm.record_slots(T, sk_tiles=sk_tiles, sk_units=G)
    L = sk_tiles * num_kb
    pieces_per_tile = {}
    for c, u in enumerate(units[:G]):
        assert 1 <= len(u) <= 3
        assert [it[0] for it in u] == list(range(3 * c + len(u) - 1, 3 * c - 1, -1))   # last tile first
        assert u[0][4] == 0                             # every unit starts at k-block 0 of a tile
        kb = sum(it[5] - it[4] for it in u)
        assert kb in (L // G, -(-L // G))               # even shares, to within one k-block
        assert kb >= num_kb                             # at least a tile's worth each
        for it in u:
            pieces_per_tile[it[1]] = pieces_per_tile.get(it[1], 0) + 1
    assert max(pieces_per_tile.values()) <= 2
    # static assignment: cluster c runs units c, c + G, ...; every cluster ends
    # up with the same number of k-blocks to within one
    load = [0] * G
    for u, its in enumerate(units):
        load[u % G] += sum(it[5] - it[4] for it in its)
    assert max(load) - min(load) <= 1
    assert sum(load) == T * num_kb


def test_grouped_items_hand_worked():
    """Problems (300, 600), (0, 512), (128, 100) with 128 x 256 tiles and
    GROUP_SIZE_M = 2: the first has a 3 x 3 tile grid (rows 0-1 walked column
    by column, then row 2), the second none, the third one tile."""
    got = sm.grouped_items([(300, 600), (0, 512), (128, 100)], 128, 256, 2)
    assert got == [(0, 0, 0), (0, 1, 0), (0, 0, 1), (0, 1, 1), (0, 0, 2), (0, 1, 2),
                   (0, 2, 0), (0, 2, 1), (0, 2, 2), (2, 0, 0)]


def test_grouped_items_longest_first_hand_worked():
    """Three one-tile problems with 2, 5 and 5 k-blocks and one with 3: the
    5s first in their given order, then the 3, then the 2."""
    got = sm.grouped_items([(1, 8), (1, 8), (1, 8), (1, 8)], 128, 256, 8, kb=[2, 5, 5, 3])
    assert got == [(1, 0, 0), (2, 0, 0), (3, 0, 0), (0, 0, 0)]


@pytest.mark.parametrize("seed", range(5))
def test_grouped_items_cover_every_problem_tile_once(seed):
    rng = random.Random(seed)
    probs = [(rng.choice([0, 1, 127, 128, 129, 700]), rng.choice([0, 8, 256, 264, 1000])) for _ in range(12)]
    items = sm.grouped_items(probs, 256, 256, 8)
    want = {(g, tm, tn) for g, (M, N) in enumerate(probs) if M and N
            for tm in range(sm.cdiv(M, 256)) for tn in range(sm.cdiv(N, 256))}
    assert len(items) == len(want) and set(items) == want
    # problems in order, each a contiguous run
    gs = [g for g, _, _ in items]
    assert gs == sorted(gs)


def test_grouped_workload_model_predicts_clc_ahead_of_static():
    """The 64-problem grouped workload in the scheduler model (CTA pairs: 16
    tiles per problem, 76 resident clusters, a tile costing its k-blocks
    plus 6): the static stride finishes last, CLC's first-come order ends
    near the even split, and listing the problems most k-blocks first brings
    both closer to it."""
    import workloads as wl
    ps = wl.bf16_grouped_vark()
    G = 76

    def costs(order):
        return [-(-ps[g].K // 64) + 6 for g in order for _ in range(16)]

    def static_makespan(c):
        load = [0.0] * G
        for w, x in enumerate(c):
            load[w % G] += x
        return max(load)

    def clc_makespan(c):
        events, _, _ = sm.clc_replay(len(c), G, cost=lambda w: float(c[w]))
        end = {}
        # replay order: a cluster's tiles run back to back, so its finish is the sum of its costs
        for w, cluster, _ in events:
            end[cluster] = end.get(cluster, 0.0) + c[w]
        return max(end.values())

    given = list(range(len(ps)))
    longest = sorted(given, key=lambda g: -ps[g].K)
    even = sum(costs(given)) / G
    st, cl = static_makespan(costs(given)), clc_makespan(costs(given))
    st_l, cl_l = static_makespan(costs(longest)), clc_makespan(costs(longest))
    assert st > cl > even and st_l > cl_l >= even
    assert cl_l < cl and st_l < st
    assert cl < 1.1 * even and cl_l < 1.02 * even and st > 1.2 * even
