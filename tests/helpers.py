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


def compare_full(x: wl.Inputs, C: torch.Tensor):
    p = x.problem
    ref, ref_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, dequant(x))
    return og.rel_err(C.double().cpu().numpy(), ref, ref_abs, out_u(p.dtype))


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


def compare_sampled(x: wl.Inputs, C: torch.Tensor, tile_m: int, tile_n: int, seed=0):
    p = x.problem
    ii, jj = sample_positions(p.M, p.N, tile_m, tile_n, seed=seed)
    ref, ref_abs = og.gemm_sampled(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, ii, jj, dequant(x))
    got = C.double().cpu().numpy()[ii, jj]
    return og.rel_err(got, ref, ref_abs, out_u(p.dtype))


def check_records(records, info, sched: int, K: int, group_m: int = 8):
    """Per-work-item records against what the schedulers must do (bit-exact)."""
    T, Tm, Tn, cg = int(info.tiles), int(info.tiles_m), int(info.tiles_n), int(info.cta_group)
    W, F, split = int(info.work_items), int(info.full_work), int(info.split)
    G = int(info.grid_ctas) // cg
    num_kb = -(-int(K) // int(info.tile_k))
    items = osched.work_items(T, F, split, split_k=bool(info.split_k), num_kb=num_kb,
                              part_kb=int(info.part_kb) if info.split_k else None)
    assert len(items) == W
    cover = {}
    for w, t_order, n_off, n_len, k0, k1 in items:
        r = records[w]
        assert r.visits == cg, f"work item {w} stored {r.visits} times"
        tm, tn = osched.swizzle(t_order, Tm, Tn, group_m)
        assert (r.tile, r.n_off, r.n_len) == (tm * Tn + tn, n_off, n_len), w
        assert (r.kb_begin, r.kb_end) == (k0, k1), w
        cover.setdefault(r.tile, []).append((r.kb_begin, r.kb_end, r.n_off, r.n_len))
    # the items partition every tile (columns x k-blocks) exactly once
    assert sorted(cover) == list(range(T))
    for t, parts in cover.items():
        cells = sum((k1 - k0) * n for k0, k1, _, n in parts)
        kb_total = max(k1 for _, k1, _, _ in parts)
        assert cells == 256 * kb_total, t
    by_work = {w: (records[w].owner, records[w].iter) for w in range(W)}
    if sched == pts.GEMM_SCHED_STATIC:
        want = {w: (c, it) for w, c, it in osched.static_assignment(W, G)}
        assert by_work == want
    elif sched == pts.GEMM_SCHED_NONPERSISTENT:
        want = {w: (c, it) for w, c, it in osched.nonpersistent_assignment(W)}
        assert by_work == want
    else:
        # CLC: a cluster's first item is its own id; its later items were
        # cancelled clusters, each run exactly once; iterations are 0..n-1
        per_owner = {}
        for w, (owner, it) in by_work.items():
            if it == 0:
                assert owner == w
            per_owner.setdefault(owner, []).append(it)
        for owner, its in per_owner.items():
            assert sorted(its) == list(range(len(its))), owner
    return by_work
