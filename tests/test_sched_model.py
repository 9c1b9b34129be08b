"""Pins for the scheduler model (host logic, no GPU).

The model states what each scheduler must do; these tests check it against
hand-worked orders, closed forms of the grouped order at its extremes, and the
coverage invariant ("Neither mode creates additional independent work at the
tail of a grid": every tile is done exactly once).
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
    # 5 tiles of 8 k-blocks, 4 whole, the fifth cut in two: columns 0-127 and 128-255
    assert sm.work_items(5, 4, 2, num_kb=8) == [
        (0, 0, 0, 256, 0, 8), (1, 1, 0, 256, 0, 8), (2, 2, 0, 256, 0, 8), (3, 3, 0, 256, 0, 8),
        (4, 4, 0, 128, 0, 8), (5, 4, 128, 128, 0, 8)]
    assert [i[2:4] for i in sm.work_items(2, 0, 4)[:4]] == [(0, 64), (64, 64), (128, 64), (192, 64)]
    # the same tile cut along K in three: k-blocks 0-2, 3-5, 6-9
    assert sm.work_items(5, 4, 3, split_k=True, num_kb=10)[4:] == [
        (4, 4, 0, 256, 0, 3), (5, 4, 0, 256, 3, 6), (6, 4, 0, 256, 6, 10)]
    # uneven K parts: a short first part (25 k-blocks) and a long last one (39)
    assert sm.work_items(5, 4, 2, split_k=True, num_kb=64, part_kb=25)[4:] == [
        (4, 4, 0, 256, 0, 25), (5, 4, 0, 256, 25, 64)]
    with pytest.raises(ValueError):      # parts must leave the last one at least a k-block
        sm.work_items(5, 4, 3, split_k=True, num_kb=10, part_kb=5)


@pytest.mark.parametrize("T,F,s,k,a", [(512, 456, 2, False, None), (8, 0, 4, False, None),
                                       (528, 456, 2, False, None), (150, 150, 1, False, None),
                                       (800, 760, 2, False, None), (512, 456, 2, True, None),
                                       (256, 228, 3, True, None), (800, 760, 4, True, None), (8, 0, 4, True, None),
                                       (512, 456, 2, True, 2), (256, 228, 3, True, 1)])
def test_work_items_partition_every_tile(T, F, s, k, a):
    num_kb = 7
    items = sm.work_items(T, F, s, split_k=k, num_kb=num_kb, part_kb=a)
    assert [i[0] for i in items] == list(range(F + s * (T - F)))
    cells = {}
    for _, t, off, n, k0, k1 in items:
        assert k1 > k0
        cells.setdefault(t, []).append((off, n, k0, k1))
    for t in range(T):
        got = set()
        for off, n, k0, k1 in cells[t]:
            new = {(c, kb) for c in range(off, off + n) for kb in range(k0, k1)}
            assert not (got & new)                      # nothing computed twice
            got |= new
        assert got == {(c, kb) for c in range(256) for kb in range(num_kb)}
