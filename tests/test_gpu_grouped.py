"""GPU parity of the grouped launch (several independent GEMMs, one launch).

Every problem's C is compared with the oracle element by element (small
shapes) or on sampled outputs (the 64-problem workload), and must be
bit-identical to the same problem run alone through gemm_run with the same
tiles; the tile records must match the grouped work-id model and each
scheduler's assignment bit-exactly.
"""
import ctypes

import numpy as np
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og
from oracle import sched as osched

from helpers import TOL, compare_full, compare_sampled

pytestmark = pytest.mark.gpu

SCHEDS = [pts.GEMM_SCHED_NONPERSISTENT, pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC]

# ragged shapes, an empty problem, K = 0, N = 8, a single k-block
SMALL = [(300, 520, 208), (0, 64, 64), (128, 256, 0), (257, 8, 1008), (64, 1000, 16), (512, 512, 512),
         (1, 264, 96)]


def _inputs(shapes, dtype, seed0):
    return [wl.custom(M, N, K, dtype, "uniform", seed=seed0 + i) for i, (M, N, K) in enumerate(shapes)]


def _device(xs):
    out = []
    for x in xs:
        p = x.problem
        C = torch.full((p.M, p.N), float("nan"), dtype=wl.output_torch_dtype(p.dtype), device="cuda")
        out.append((x.A.cuda(), x.B.cuda(), C))
    return out


def _problems(xs, dev):
    return [(x.problem.M, x.problem.N, x.problem.K, A, B, C, x.scale_a, x.scale_b)
            for x, (A, B, C) in zip(xs, dev)]


def _check_grouped_records(h, xs, info, sched, group_m=8, longest_first=True):
    cg = int(info.cta_group)
    W = int(info.work_items)
    kelems = int(info.tile_k)
    st, recs, dev = pts.gemm_read_debug(h, W)
    assert st == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
    kb = [-(-x.problem.K // kelems) for x in xs] if longest_first else None
    items = osched.grouped_items([(x.problem.M, x.problem.N) for x in xs], 128 * cg, 256, group_m, kb)
    assert len(items) == W == int(info.tiles) == int(info.units)
    for w, (g, tm, tn) in enumerate(items):
        r = recs[w]
        p = xs[g].problem
        Tn = -(-p.N // 256)
        assert r.visits == cg, f"work item {w} stored {r.visits} times"
        assert (r.group, r.tile, r.n_off, r.n_len) == (g, tm * Tn + tn, 0, 256), w
        assert (r.kb_begin, r.kb_end) == (0, -(-p.K // kelems)), w
    by_work = [(recs[w].owner, recs[w].iter) for w in range(W)]
    G = int(info.grid_ctas) // cg
    if sched == pts.GEMM_SCHED_STATIC:
        assert by_work == [(w % G, w // G) for w in range(W)]
    elif sched == pts.GEMM_SCHED_NONPERSISTENT:
        assert by_work == [(w, 0) for w in range(W)]
    else:
        per_owner = {}
        for w, (owner, it) in enumerate(by_work):
            if it == 0:
                assert owner == w
            per_owner.setdefault(owner, []).append(it)
        for owner, its in per_owner.items():
            assert sorted(its) == list(range(len(its))), owner


@pytest.fixture(scope="module", params=[1, 2], ids=["cg1", "cg2"])
def handles(request):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cg = request.param
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, debug_flags=pts.GEMM_DEBUG_RECORDS))
    # one problem at a time, whole tiles only: the same tiles as the grouped launch
    h1 = pts.gemm_create(0, pts.make_opts(cta_group=cg, split=1, split_k=-1))
    yield h, h1, cg
    pts.gemm_destroy(h)
    pts.gemm_destroy(h1)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16, wl.E4M3])
@pytest.mark.parametrize("sched", SCHEDS)
def test_grouped_small_problems(handles, dtype, sched):
    h, h1, cg = handles
    shapes = [(M, N, K if dtype != wl.E4M3 else (K + 15) // 16 * 16) for M, N, K in SMALL]
    xs = _inputs(shapes, dtype, seed0=900 + 10 * dtype)
    dev = _device(xs)
    probs = _problems(xs, dev)
    pts.gemm_run_grouped(h, probs, dtype, sched)
    info = pts.gemm_query_grouped(h, probs, dtype, sched)
    assert int(info.cta_group) == cg
    _check_grouped_records(h, xs, info, sched)
    for x, (A, B, C) in zip(xs, dev):
        p = x.problem
        if p.M == 0 or p.N == 0:
            continue
        if p.K == 0:
            assert torch.count_nonzero(C).item() == 0
            continue
        err = compare_full(x, C)
        assert err <= TOL[dtype], f"{p.name}: rel err {err}"
        # the same problem alone, same tiles: the same bits
        C1 = torch.full_like(C, float("nan"))
        pts.gemm_run(h1, p.M, p.N, p.K, A, B, C1, dtype, sched, x.scale_a, x.scale_b)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), C1.view(torch.int16)), p.name


@pytest.mark.parametrize("sched", SCHEDS)
def test_grouped_given_order(sched):
    """group_order 2: the problems' tiles in the caller's order."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    xs = _inputs([(256, 512, 64), (300, 264, 1024), (128, 256, 0), (512, 256, 512)], wl.BF16, 80)
    dev = _device(xs)
    probs = _problems(xs, dev)
    h = pts.gemm_create(0, pts.make_opts(cta_group=2, group_order=2, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        pts.gemm_run_grouped(h, probs, wl.BF16, sched)
        info = pts.gemm_query_grouped(h, probs, wl.BF16, sched)
        _check_grouped_records(h, xs, info, sched, longest_first=False)
        for x, (_, _, C) in zip(xs, dev):
            if x.problem.K:
                assert compare_full(x, C) <= TOL[wl.BF16]
            else:
                assert torch.count_nonzero(C).item() == 0
    finally:
        pts.gemm_destroy(h)


def test_grouped_table_reuse_and_change(handles):
    """Lists X, Y, X, X (the last after new values in X's inputs) on one
    stream: an unchanged list reuses its table, a changed one gets the other
    slot; every result is right."""
    h, _, cg = handles
    xs_x = _inputs([(256, 512, 128), (384, 256, 64)], wl.BF16, 50)
    xs_y = _inputs([(128, 264, 256), (640, 512, 32), (8, 8, 8)], wl.BF16, 60)
    dx, dy = _device(xs_x), _device(xs_y)
    for xs, d in ((xs_x, dx), (xs_y, dy), (xs_x, dx)):
        for _, _, C in d:
            C.fill_(float("nan"))
        pts.gemm_run_grouped(h, _problems(xs, d), wl.BF16, pts.GEMM_SCHED_CLC)
        assert pts.gemm_check(h)[0] == 0
        for x, (_, _, C) in zip(xs, d):
            assert compare_full(x, C) <= TOL[wl.BF16]
    # new values in the same buffers: the reused table points at them
    xs_x2 = _inputs([(256, 512, 128), (384, 256, 64)], wl.BF16, 70)
    for x2, (A, B, C) in zip(xs_x2, dx):
        A.copy_(x2.A.cuda())
        B.copy_(x2.B.cuda())
        C.fill_(float("nan"))
    pts.gemm_run_grouped(h, _problems(xs_x2, dx), wl.BF16, pts.GEMM_SCHED_STATIC)
    assert pts.gemm_check(h)[0] == 0
    for x2, (_, _, C) in zip(xs_x2, dx):
        assert compare_full(x2, C) <= TOL[wl.BF16]


def test_grouped_empty_lists_launch_nothing(handles):
    h, _, _ = handles
    assert pts.gemm_run_grouped(h, [], wl.BF16, pts.GEMM_SCHED_STATIC) == 0
    C = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    assert pts.gemm_run_grouped(h, [(0, 64, 64, 0, 0, C)], wl.BF16, pts.GEMM_SCHED_CLC) == 0
    info = pts.gemm_query_grouped(h, [(0, 64, 64, 0, 0, C)], wl.BF16, pts.GEMM_SCHED_CLC)
    assert info.tiles == 0 and info.grid_ctas == 0


# the capture below is meant to stay empty (the call refuses a capturing stream)
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_grouped_invalid_arguments(handles):
    h, _, _ = handles
    lib = pts.load()
    x = wl.custom(128, 256, 64, wl.BF16, "uniform", seed=3)
    A, B = x.A.cuda(), x.B.cuda()
    C = torch.empty(128, 256, dtype=torch.bfloat16, device="cuda")
    good = (128, 256, 64, A, B, C)

    def status(probs, dtype=wl.BF16, sched=pts.GEMM_SCHED_STATIC, count=None):
        g = pts.gemm.group_array(probs)
        n = g.count if count is None else count
        return lib.gemm_run_grouped(h, g.arr, n, dtype, sched, None)

    bad = pts.gemm.GEMM_ERR_INVALID_ARG
    assert status([good]) == 0
    assert status([good], count=-1) == bad
    assert status([good], count=pts.gemm.GEMM_GROUPED_MAX_PROBLEMS + 1) == bad
    assert lib.gemm_run_grouped(h, None, 1, wl.BF16, 1, None) == bad
    assert status([good], dtype=3) == bad
    assert status([good], sched=3) == bad
    assert status([good, (128, 256, 60, A, B, C)]) == bad            # K % 8
    assert status([(128, 250, 64, A, B, C)]) == bad                  # N % 8
    assert status([(128, 256, 64, A.data_ptr() + 2, B, C)]) == bad   # misaligned A
    assert status([(128, 256, 64, A, B, 0)]) == bad                  # no C
    assert status([(128, 256, 64, 0, B, C)]) == bad                  # no A with K > 0
    a8 = torch.zeros(128, 64, dtype=torch.uint8, device="cuda")
    b8 = torch.zeros(256, 64, dtype=torch.uint8, device="cuda")
    assert status([(128, 256, 64, a8, b8, C, 0.0, 1.0)], dtype=wl.E4M3) == bad   # scale 0
    assert pts.gemm_check(h)[0] == 0
    # a capturing stream is refused (the table would outlive the call)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        st = lib.gemm_run_grouped(h, pts.gemm.group_array([good]).arr, 1, wl.BF16, 1, ctypes.c_void_p(s.cuda_stream))
        g.capture_end()
    assert st == bad
    torch.cuda.synchronize()


@pytest.mark.slow
@pytest.mark.parametrize("sched", SCHEDS)
def test_grouped_workload_sampled(sched):
    """The 64-problem workload of varied K, with the library's own choice of
    CTA group: records exact, four problems sampled against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    xs = [wl.make_inputs(p) for p in wl.bf16_grouped_vark()]
    dev = _device(xs)
    probs = _problems(xs, dev)
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        pts.gemm_run_grouped(h, probs, wl.BF16, sched)
        info = pts.gemm_query_grouped(h, probs, wl.BF16, sched)
        _check_grouped_records(h, xs, info, sched)
        ks = [x.problem.K for x in xs]
        pick = sorted({int(np.argmax(ks)), int(np.argmin(ks)), 17, 42})
        for i in pick:
            err = compare_sampled(xs[i], dev[i][2], int(info.tile_m), 256, seed=i)
            assert err <= TOL[wl.BF16], f"{xs[i].problem.name}: rel err {err}"
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("sched,clc_depth", [(pts.GEMM_SCHED_NONPERSISTENT, 0), (pts.GEMM_SCHED_STATIC, 0),
                                             (pts.GEMM_SCHED_CLC, 1), (pts.GEMM_SCHED_CLC, 2)])
def test_grouped_three_thousand_small_problems(sched, clc_depth):
    """3000 small ragged problems (some empty, some with K = 0) in one launch:
    the problem search takes several rounds and the scheduler's cached
    problem changes at nearly every tile.  Every C against the oracle, the
    records exactly."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    rng = np.random.default_rng(5)
    shapes = []
    for _ in range(3000):
        M = int(rng.choice([0, 1, 37, 128, 129, 300]))
        N = int(rng.choice([8, 64, 256, 264]))
        K = int(rng.choice([0, 8, 64, 200]))
        shapes.append((M, N, K))
    xs = _inputs(shapes, wl.BF16, 20000)
    dev = _device(xs)
    probs = pts.gemm.group_array(_problems(xs, dev))
    h = pts.gemm_create(0, pts.make_opts(cta_group=1, clc_depth=clc_depth, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        pts.gemm_run_grouped(h, probs, wl.BF16, sched)
        info = pts.gemm_query_grouped(h, probs, wl.BF16, sched)
        _check_grouped_records(h, xs, info, sched)
        for x, (A, B, C) in zip(xs, dev):
            p = x.problem
            if p.M == 0:
                continue
            if p.K == 0:
                assert torch.count_nonzero(C).item() == 0
                continue
            ref, ref_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, nthreads=1)
            err = og.rel_err(C.double().cpu().numpy(), ref, ref_abs, og.OUT_UNIT_ROUNDOFF[og.BF16])
            assert err <= TOL[wl.BF16], f"{p.name}: rel err {err}"
    finally:
        pts.gemm_destroy(h)
