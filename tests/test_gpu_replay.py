"""GPU parity of launches captured in a CUDA graph and replayed.

A replayed launch runs with exactly the arguments it was captured with.  The
stream-K fixup (a tile cut between two units is summed through an fp32
partial, a claim counter and a ready flag in the handle's workspace) must
therefore not depend on anything the host changes from call to call: every
launch finds its counters and flags at zero and leaves them at zero.  These
tests replay such launches several times and compare every replay's C with
the oracle, on the elements of the cut tiles (where a stale partial would
show) as well as on the usual sample of the whole output.

The tile boundary of "Choosing between static and CLC scheduling" is the
guide: however the work is handed out, each output element is computed
exactly once, replay or not.
"""
import numpy as np
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og
from oracle import sched as osched

from helpers import TOL, dequant, out_u, record_parity, sample_positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def cut_tile_positions(info, M, N, K, n_random=256, seed=0):
    """Element positions inside the tiles that the stream-K share cuts in two:
    the four corners of each, the first and last row and column of each, and
    random elements (the tile is given by the scheduler model's work items)."""
    T, Tm, Tn = int(info.tiles), int(info.tiles_m), int(info.tiles_n)
    BM, BN = int(info.tile_m), int(info.tile_n)
    num_kb = -(-K // int(info.tile_k))
    units = osched.work_units(T, 1, num_kb=num_kb, sk_tiles=int(info.sk_tiles), sk_units=int(info.sk_units))
    cut = sorted({it[1] for u in units for it in u if (it[4], it[5]) != (0, num_kb)})
    assert cut, "the plan cuts no tile: nothing for the fixup to do"
    rng = np.random.default_rng(seed)
    ii, jj = [], []
    for t in cut:
        tm, tn = osched.swizzle(t, Tm, Tn, 8)
        r0, c0 = tm * BM, tn * BN
        r1, c1 = min(r0 + BM, M) - 1, min(c0 + BN, N) - 1
        rows = np.arange(r0, r1 + 1)
        cols = np.arange(c0, c1 + 1)
        ii += [np.array([r0, r0, r1, r1]), rows, rows, np.full(cols.size, r0), np.full(cols.size, r1),
               rng.integers(r0, r1 + 1, n_random)]
        jj += [np.array([c0, c1, c0, c1]), np.full(rows.size, c0), np.full(rows.size, c1), cols, cols,
               rng.integers(c0, c1 + 1, n_random)]
    return np.concatenate(ii).astype(np.int64), np.concatenate(jj).astype(np.int64), len(cut)


def _check_positions(x, C, ii, jj, what):
    p = x.problem
    ref, ref_abs = og.gemm_sampled(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, ii, jj, dequant(x))
    got = C.double().cpu().numpy()[ii, jj]
    err = og.rel_err(got, ref, ref_abs, out_u(p.dtype))
    record_parity(what, p, got, ref, ref_abs)
    assert err <= TOL[p.dtype], f"{what}: rel err {err}"


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", [pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC, pts.GEMM_SCHED_NONPERSISTENT])
def test_captured_stream_k_gemm_replayed_three_times(cg, sched):
    """One fp16 4096^3 GEMM with the stream-K share, captured once and replayed
    three times.  Before each replay the captured A and B buffers receive new
    seeded inputs and C is overwritten with NaN, so a partial left over from an
    earlier replay holds the wrong numbers; every replay must match its own
    inputs' oracle on every cut tile."""
    p = wl.fp16_4096_ksweep([4096])[0]
    xs = [wl.make_inputs(wl.Problem(p.name, p.M, p.N, p.K, p.dtype, p.dist, p.seed + 100 * r)) for r in range(3)]
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, split_k=1))
    s = torch.cuda.Stream()
    try:
        info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, sched)
        assert info.split_k == 1
        A, B = xs[0].A.cuda(), xs[0].B.cuda()
        C = torch.empty(p.M, p.N, dtype=torch.float16, device="cuda")
        torch.cuda.synchronize()
        pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, 1.0, 1.0, s)   # grows the workspace
        assert pts.gemm_check(h, s)[0] == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, 1.0, 1.0, s)
        ii, jj, ncut = cut_tile_positions(info, p.M, p.N, p.K)
        ri, rj = sample_positions(p.M, p.N, int(info.tile_m), int(info.tile_n), n_random=2048, seed=3)
        for r, x in enumerate(xs):
            with torch.cuda.stream(s):
                A.copy_(x.A, non_blocking=False)
                B.copy_(x.B, non_blocking=False)
                C.fill_(float("nan"))
                g.replay()
            st, dev = pts.gemm_check(h, s)
            assert st == 0, f"replay {r}: {pts.gemm_status_string(st)}, device word {dev:#x}"
            _check_positions(x, C, ii, jj, f"replay {r}, {ncut} cut tiles")
            _check_positions(x, C, ri, rj, f"replay {r}, sampled")
        del g
    finally:
        pts.gemm_destroy(h)


def test_graph_with_the_same_stream_k_gemm_twice():
    """Two launches of one stream-K GEMM inside one graph, on two input sets
    into two outputs: the second launch of each replay starts from the
    counters the first left; new inputs before every replay."""
    p = wl.fp16_4096_ksweep([2048])[0]
    h = pts.gemm_create(0, pts.make_opts(cta_group=2, split_k=1))
    s = torch.cuda.Stream()
    try:
        info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, pts.GEMM_SCHED_STATIC)
        sets = [[wl.make_inputs(wl.Problem(p.name, p.M, p.N, p.K, p.dtype, p.dist, p.seed + 10 * r + n))
                 for n in range(2)] for r in range(2)]
        dev = [(sets[0][n].A.cuda(), sets[0][n].B.cuda(), torch.empty(p.M, p.N, dtype=torch.float16, device="cuda"))
               for n in range(2)]
        torch.cuda.synchronize()
        A0, B0, C0 = dev[0]
        pts.gemm_run(h, p.M, p.N, p.K, A0, B0, C0, p.dtype, pts.GEMM_SCHED_STATIC, 1.0, 1.0, s)
        assert pts.gemm_check(h, s)[0] == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for A, B, C in dev:
                pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_STATIC, 1.0, 1.0, s)
        ii, jj, _ = cut_tile_positions(info, p.M, p.N, p.K)
        for r in range(2):
            with torch.cuda.stream(s):
                for (A, B, C), x in zip(dev, sets[r]):
                    A.copy_(x.A)
                    B.copy_(x.B)
                    C.fill_(float("nan"))
                g.replay()
            assert pts.gemm_check(h, s)[0] == 0
            for n, ((_, _, C), x) in enumerate(zip(dev, sets[r])):
                _check_positions(x, C, ii, jj, f"replay {r}, launch {n}")
        del g
    finally:
        pts.gemm_destroy(h)


@pytest.mark.slow
def test_bench_step_replayed_matches_oracle():
    """bench.py's own step (the 32 GEMMs of the fp16 4096 K sweep, library
    defaults, static scheduler), captured as bench.py --graph captures it and
    replayed twice; the K = 3072 and K = 4096 outputs (CTA pairs with the
    stream-K share) are checked against the oracle after each replay, and
    the K = 2048 one (CTA pairs) and the K = 128 one (single CTAs), both with
    their last wave's tiles in column halves, on a sample."""
    import bench
    problems = wl.fp16_4096_ksweep()
    checked = {128, 2048, 3072, 4096}
    xs, bufs = {}, []
    gen = torch.Generator(device="cuda").manual_seed(12)
    for q in problems:
        if q.K in checked:
            xs[q.K] = wl.make_inputs(q)
            A, B = xs[q.K].A.cuda(), xs[q.K].B.cuda()
        else:
            A = torch.randn(q.M, q.K, device="cuda", generator=gen).to(torch.float16)
            B = torch.randn(q.N, q.K, device="cuda", generator=gen).to(torch.float16)
        bufs.append((A, B, torch.empty(q.M, q.N, dtype=torch.float16, device="cuda")))
    torch.cuda.synchronize()
    h = pts.gemm_create(0, pts.make_opts(cta_group=0, epilogue=0, split_k=0))
    s = torch.cuda.Stream()
    try:
        # the step holds launches with the stream-K share and with tail halves
        for K in (3072, 4096):
            assert pts.gemm_query(h, 4096, 4096, K, wl.F16, pts.GEMM_SCHED_STATIC).split_k == 1
        assert pts.gemm_query(h, 4096, 4096, 2048, wl.F16, pts.GEMM_SCHED_STATIC).tail_tiles > 0
        with torch.cuda.stream(s):
            bench.sweep_pass(pts, h, bufs, problems, pts.GEMM_SCHED_STATIC, s)
        assert pts.gemm_check(h, s)[0] == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bench.sweep_pass(pts, h, bufs, problems, pts.GEMM_SCHED_STATIC, s)
        for r in range(2):
            with torch.cuda.stream(s):
                for q, (A, B, C) in zip(problems, bufs):
                    if q.K in checked:
                        if r > 0:   # new inputs, so that a stale partial would show
                            xs[q.K] = wl.make_inputs(wl.Problem(q.name, q.M, q.N, q.K, q.dtype, q.dist, q.seed + 7 * r))
                            A.copy_(xs[q.K].A)
                            B.copy_(xs[q.K].B)
                        C.fill_(float("nan"))
                g.replay()
            assert pts.gemm_check(h, s)[0] == 0
            for q, (_, _, C) in zip(problems, bufs):
                if q.K not in checked:
                    continue
                info = pts.gemm_query(h, q.M, q.N, q.K, q.dtype, pts.GEMM_SCHED_STATIC)
                ii, jj = sample_positions(q.M, q.N, int(info.tile_m), int(info.tile_n), n_random=2048, seed=r)
                if info.split_k:
                    ci, cj, _ = cut_tile_positions(info, q.M, q.N, q.K, n_random=64)
                    ii, jj = np.concatenate([ii, ci]), np.concatenate([jj, cj])
                _check_positions(xs[q.K], C, ii, jj, f"bench step replay {r}, K={q.K}")
        del g
    finally:
        pts.gemm_destroy(h)
