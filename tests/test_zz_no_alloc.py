"""gemm_run_noalloc, the entry point that allocates nothing, against gemm_run.

Some callers cannot allocate device memory when they need a GEMM: runtimes
that reserve all device memory at start-up and refuse later allocations, and
latency-critical loops that cannot accept the implicit synchronisation that
cudaMalloc / cudaFree may perform.  gemm_run_noalloc serves them: it needs no
handle and keeps the kernel's scratch (status block, per-tile coverage
records) in a static device array shared by all calls.

For problems smaller than one wave of resident clusters both entry points
take the same plan (CTA group, ring depth, column slices, no stream-K share),
so gemm_run_noalloc must return exactly the bits gemm_run returns, and both
must meet the oracle's bound.  The same holds past one wave while gemm_run
takes no stream-K share (short tiles): both then run a partial last wave as
column halves.  Two calls in a row, on problems of different
sizes, check that the shared scratch is cleared between calls (the second
call would otherwise find the first call's tile records).  This file is
collected last on purpose.
"""
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og

from helpers import TOL, compare_sampled, dequant, out_u

pytestmark = pytest.mark.gpu

SCHEDS = [pts.GEMM_SCHED_NONPERSISTENT, pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC]
# two sub-wave problems of different sizes (K a multiple of 16, so every dtype takes them)
SHAPES = [(1000, 1032, 512), (520, 264, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _inputs(dtype, i):
    M, N, K = SHAPES[i]
    dist = "normal" if dtype == wl.E4M3 else "uniform"
    return wl.make_inputs(wl.Problem("noalloc", M, N, K, dtype, dist, 41 + 7 * dtype + i))


def _run_existing(h, x, sched):
    p = x.problem
    A, B = x.A.cuda(), x.B.cuda()
    C = torch.full((p.M, p.N), float("nan"), dtype=wl.output_torch_dtype(p.dtype), device="cuda")
    pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, x.scale_a, x.scale_b)
    assert pts.gemm_check(h)[0] == 0
    return A, B, C


def _bits(C):
    return C.view(torch.int16)


@pytest.mark.parametrize("sched", SCHEDS, ids=["nonpersistent", "static", "clc"])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16, wl.E4M3], ids=["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("cg", [1, 2])
def test_noalloc_matches_gemm_run_on_two_calls_in_a_row(cg, dtype, sched):
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg))
    try:
        for i in range(len(SHAPES)):
            x = _inputs(dtype, i)
            p = x.problem
            info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, sched)
            assert info.split_k == 0 and info.cta_group == cg   # the plan gemm_run_noalloc takes too
            A, B, C_existing = _run_existing(h, x, sched)
            C = torch.full((p.M, p.N), float("nan"), dtype=C_existing.dtype, device="cuda")
            st, dev = pts.gemm_run_noalloc(p.M, p.N, p.K, A, B, C, p.dtype, sched, x.scale_a, x.scale_b,
                                           cta_group=cg, check=True)
            assert st == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
            assert dev == 0
            assert torch.equal(_bits(C), _bits(C_existing)), f"call {i}: not bit-identical to gemm_run"
            ref, ref_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype, dequant(x))
            err = og.rel_err(C.double().cpu().numpy(), ref, ref_abs, out_u(p.dtype))
            assert err <= TOL[p.dtype], err
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("sched", SCHEDS, ids=["nonpersistent", "static", "clc"])
@pytest.mark.parametrize("cg", [1, 2])
def test_noalloc_partial_last_wave(cg, sched):
    """A problem of several waves (fp16 4096^2 x 256) whose partial last wave
    the persistent schedulers run as column halves, in both entry points:
    gemm_run_noalloc gives gemm_run's bits, its coverage records are exact,
    and a sample meets the oracle's bound."""
    x = wl.make_inputs(wl.Problem("noalloc_tail", 4096, 4096, 256, wl.F16, "normal_sqrtk", 45 + cg))
    p = x.problem
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg))
    try:
        info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, sched)
        assert info.split_k == 0 and info.tiles > info.max_active_clusters
        assert (int(info.tail_tiles) > 0) == (sched != pts.GEMM_SCHED_NONPERSISTENT)
        A, B, C_existing = _run_existing(h, x, sched)
    finally:
        pts.gemm_destroy(h)
    C = torch.full((p.M, p.N), float("nan"), dtype=C_existing.dtype, device="cuda")
    st, dev = pts.gemm_run_noalloc(p.M, p.N, p.K, A, B, C, p.dtype, sched, cta_group=cg, check=True)
    assert st == 0 and dev == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
    assert torch.equal(_bits(C), _bits(C_existing))
    err = compare_sampled(x, C, int(info.tile_m), int(info.tile_n))
    assert err <= TOL[p.dtype], err


def test_noalloc_asynchronous_call_matches():
    """Without a status pointer the call returns after the launch; two such
    calls in a row give gemm_run's bits."""
    x = wl.custom(384, 512, 256, wl.BF16, "uniform", 43)
    p = x.problem
    h = pts.gemm_create(0, pts.make_opts(cta_group=1))
    try:
        A, B, C_existing = _run_existing(h, x, pts.GEMM_SCHED_STATIC)
    finally:
        pts.gemm_destroy(h)
    for _ in range(2):
        C = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st, _ = pts.gemm_run_noalloc(p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_STATIC)
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(_bits(C), _bits(C_existing))


def test_noalloc_rejects_problems_beyond_its_scratch():
    """More output tiles than the static scratch holds: rejected before any launch."""
    M, N, K = 128 * 129, 256 * 128, 8          # 16 512 tiles of 128 x 256 > 16 384
    assert (M // 128) * (N // 256) > pts.gemm.GEMM_NOALLOC_MAX_WORK_ITEMS
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    st, _ = pts.gemm_run_noalloc(M, N, K, A, B, C, pts.GEMM_BF16, pts.GEMM_SCHED_STATIC, check=True)
    assert st == pts.gemm.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert not C.any()
    del A, B, C
    torch.cuda.empty_cache()
