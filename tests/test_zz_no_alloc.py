"""gemm_run_noalloc, the entry point that allocates nothing, against gemm_run.

Some callers cannot allocate device memory when they need a GEMM: runtimes
that reserve all device memory at start-up and refuse later allocations, and
latency-critical loops that cannot accept the implicit synchronisation that
cudaMalloc / cudaFree may perform.  gemm_run_noalloc serves them: it needs no
handle and keeps the kernel's scratch (status block, per-tile coverage
records) in a static device array shared by all calls.

Two calls in a row, on problems of different sizes, must each match what
gemm_run computes on the same inputs within the parity tolerance; the second
call would trip over the first call's tile records if the shared scratch were
not cleared between calls.  This file is collected last on purpose.
"""
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og

pytestmark = pytest.mark.gpu

TOL = 2e-3   # the fp16/bf16 parity bound of the GPU tests


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _run_existing(h, x, sched):
    p = x.problem
    A, B = x.A.cuda(), x.B.cuda()
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched)
    assert pts.gemm_check(h)[0] == 0
    return A, B, C


@pytest.mark.parametrize("cg", [1, 2])
def test_noalloc_matches_gemm_run_on_two_calls_in_a_row(cg):
    xs = [wl.custom(1000, 1032, 520, wl.BF16, "uniform", 41),
          wl.custom(520, 264, 1024, wl.BF16, "uniform", 42)]
    scheds = [pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC]
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg))
    try:
        for x, sched in zip(xs, scheds):
            p = x.problem
            A, B, C_existing = _run_existing(h, x, sched)
            C = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            st, dev = pts.gemm_run_noalloc(p.M, p.N, p.K, A, B, C, p.dtype, sched, cta_group=cg, check=True)
            assert st == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
            assert dev == 0
            _, C_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype)
            err = og.rel_err(C.double().cpu().numpy(), C_existing.double().cpu().numpy(), C_abs)
            assert err <= TOL, err
    finally:
        pts.gemm_destroy(h)


def test_noalloc_asynchronous_call_matches():
    """Without a status pointer the call returns after the launch."""
    x = wl.custom(384, 512, 256, wl.BF16, "uniform", 43)
    p = x.problem
    h = pts.gemm_create(0, pts.make_opts(cta_group=1))
    try:
        A, B, C_existing = _run_existing(h, x, pts.GEMM_SCHED_STATIC)
    finally:
        pts.gemm_destroy(h)
    C = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        st, _ = pts.gemm_run_noalloc(p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_STATIC)
        assert st == 0
    torch.cuda.synchronize()
    _, C_abs = og.gemm(p.M, p.N, p.K, x.bits("A"), x.bits("B"), p.dtype)
    assert og.rel_err(C.double().cpu().numpy(), C_existing.double().cpu().numpy(), C_abs) <= TOL


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
