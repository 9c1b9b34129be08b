"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
pick sample positions, compare with the oracle, check tile records."""
from __future__ import annotations

import numpy as np
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og
from oracle import sched as osched

TOL = {wl.F16: 2e-3, wl.BF16: 2e-3, wl.E4M3: 3e-2}
SCHED_NAMES = {0: "nonpersistent", 1: "static", 2: "clc"}


def run_device(h, x: wl.Inputs, sched: int, stream=None) -> torch.Tensor:
    p = x.problem
    A, B = x.A.cuda(), x.B.cuda()
    C = torch.full((p.M, p.N), float("nan"), dtype=wl.output_torch_dtype(p.dtype), device="cuda")
    pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, x.scale_a, x.scale_b, stream)
    return C


def dequant(x: wl.Inputs) -> float:
    return 1.0 / (float(x.scale_a) * float(x.scale_b)) if x.problem.dtype == wl.E4M3 else 1.0


def out_u(dtype: int) -> float:
    """Unit roundoff of the output format (fp16 C for fp16 in, bf16 C otherwise)."""
    return og.OUT_UNIT_ROUNDOFF[og.F16 if dtype == wl.F16 else og.BF16]


# Error distribution of every parity comparison of the session (reported at
# the end of the run; written as JSON to $PTS_PARITY_REPORT when that is set).
PARITY_LOG = []


def record_parity(what: str, p, got, ref, ref_abs):
    """Log one comparison: the plain metric (no output-rounding allowance),
    the one the tests bound (with it), and percentiles of the per-element
    normalised error |C - C_ref| / (s * sum_k |a||b|)."""
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    ref_abs = np.asarray(ref_abs, np.float64).ravel()
    nz = ref_abs != 0
    e = np.abs(got[nz] - ref[nz]) / ref_abs[nz] if nz.any() else np.zeros(1)
    PARITY_LOG.append({
        "what": what, "dtype": wl.DTYPE_NAMES[p.dtype], "M": p.M, "N": p.N, "K": p.K, "elements": int(got.size),
        "plain_max": og.rel_err(got, ref, ref_abs, 0.0),
        "bounded_max": og.rel_err(got, ref, ref_abs, out_u(p.dtype)),
        "p50": float(np.percentile(e, 50)), "p99": float(np.percentile(e, 99)),
        "p999": float(np.percentile(e, 99.9)),
    })


def compare_full(x: wl.Inputs, C: torch.Tensor, what: str = "full"):
    p = x.problem
    ref, ref_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, dequant(x))
    got = C.double().cpu().numpy()
    record_parity(what, p, got, ref, ref_abs)
    return og.rel_err(got, ref, ref_abs, out_u(p.dtype))


def sample_positions(M, N, tile_m, tile_n, n_random=4096, seed=0):
    """Random elements, the four corners of every tile, the last row and column."""
    rng = np.random.default_rng(seed)
    ii = [rng.integers(0, M, n_random)]
    jj = [rng.integers(0, N, n_random)]
    r0 = np.arange(0, M, tile_m)
    c0 = np.arange(0, N, tile_n)
    R, Cc = np.meshgrid(r0, c0, indexing="ij")
    R, Cc = R.ravel(), Cc.ravel()
    r1 = np.minimum(R + tile_m - 1, M - 1)
    c1 = np.minimum(Cc + tile_n - 1, N - 1)
    ii += [R, R, r1, r1, np.full(N, M - 1), np.arange(M)]
    jj += [Cc, c1, Cc, c1, np.arange(N), np.full(M, N - 1)]
    return np.concatenate(ii).astype(np.int64), np.concatenate(jj).astype(np.int64)


def compare_sampled(x: wl.Inputs, C: torch.Tensor, tile_m: int, tile_n: int, seed=0, what: str = "sampled"):
    p = x.problem
    ii, jj = sample_positions(p.M, p.N, tile_m, tile_n, seed=seed)
    ref, ref_abs = og.gemm_sampled(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, ii, jj, dequant(x))
    got = C.double().cpu().numpy()[ii, jj]
    record_parity(what, p, got, ref, ref_abs)
    return og.rel_err(got, ref, ref_abs, out_u(p.dtype))


def check_records(records, info, sched: int, K: int, group_m: int = 8):
    """Per-work-item records against what the schedulers must do (bit-exact)."""
    T, Tm, Tn, cg = int(info.tiles), int(info.tiles_m), int(info.tiles_n), int(info.cta_group)
    W, split, BN = int(info.work_items), int(info.split), int(info.tile_n)
    G = int(info.grid_ctas) // cg
    num_kb = -(-int(K) // int(info.tile_k))
    R = int(info.tail_tiles)
    units = osched.work_units(T, split, tile_n=BN, num_kb=num_kb, sk_tiles=int(info.sk_tiles),
                              sk_units=int(info.sk_units), tail_tiles=R)
    assert len(units) == int(info.units)
    assert W == osched.record_slots(T, split, int(info.sk_tiles), int(info.sk_units), R)
    items = [it for u in units for it in u]
    used = {it[0] for it in items}
    for w in range(W):
        if w not in used:
            assert records[w].visits == 0, f"unused record slot {w} was stored"
    cover = {}
    for w, t_order, n_off, n_len, k0, k1 in items:
        r = records[w]
        assert r.visits == cg, f"work item {w} stored {r.visits} times"
        tm, tn = osched.swizzle(t_order, Tm, Tn, group_m)
        assert (r.tile, r.n_off, r.n_len) == (tm * Tn + tn, n_off, n_len), w
        assert (r.kb_begin, r.kb_end) == (k0, k1), w
        cover.setdefault(r.tile, set())
        cells = {(c, kb) for c in range(n_off, n_off + n_len, 64) for kb in range(k0, k1)}
        assert not (cover[r.tile] & cells), f"tile {r.tile} computed twice"
        cover[r.tile] |= cells
    # the items partition every tile (columns x k-blocks) exactly once
    assert sorted(cover) == list(range(T))
    full = {(c, kb) for c in range(0, BN, 64) for kb in range(num_kb)}
    assert all(cells == full for cells in cover.values())
    by_work = {it[0]: (records[it[0]].owner, records[it[0]].iter) for it in items}
    if sched == pts.GEMM_SCHED_STATIC:
        want = {}
        for c in range(G):
            it_no = 0
            for u in range(c, len(units), G):
                for it in units[u]:
                    want[it[0]] = (c, it_no)
                    it_no += 1
        assert by_work == want
    elif sched == pts.GEMM_SCHED_NONPERSISTENT:
        want = {it[0]: (u, j) for u, its in enumerate(units) for j, it in enumerate(its)}
        assert by_work == want
    else:
        # CLC: a unit runs on one cluster, its items back to back; a cluster's
        # first unit is its own id; its later units were cancelled clusters,
        # each run exactly once; every cluster's items count 0..n-1
        per_owner = {}
        for u, its in enumerate(units):
            owner, it0 = by_work[its[0][0]]
            assert [by_work[it[0]] for it in its] == [(owner, it0 + j) for j in range(len(its))], u
            if it0 == 0:
                assert owner == u
            per_owner.setdefault(owner, []).extend(range(it0, it0 + len(its)))
        for owner, its in per_owner.items():
            assert sorted(its) == list(range(len(its))), owner
    return by_work
