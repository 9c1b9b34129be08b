"""GPU parity of back-to-back launches that overlap (programmatic dependent launch).

With the launch overlap on (the default), a launch may start while the
previous kernel in the stream finishes, but it touches no global memory
before that kernel is done, so a GEMM may read the previous GEMM's output.
The test checks that contract against the oracle on a chain whose second GEMM
reads the first one's C, under every scheduler.
"""
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl

from helpers import TOL, compare_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_default_mode_chain_reads_the_previous_output():
    """C1 = A . B1, then C2 = C1 . B2 (C1 read as the next A) in the same
    stream with the launch overlap on: the second GEMM must see the first's
    complete output."""
    M, K1, N1, N2 = 640, 512, 1024, 520
    x1 = wl.custom(M, N1, K1, wl.F16, "uniform", 61)
    b2 = wl.custom(N2, 8, N1, wl.F16, "uniform", 62)        # its A (N2 x N1) is used as B2
    h = pts.gemm_create(0, pts.make_opts(overlap_launch=0))
    s = torch.cuda.Stream()
    try:
        A1, B1 = x1.A.cuda(), x1.B.cuda()
        B2 = b2.A.cuda()                                      # N2 x N1: stored N x K
        C1 = torch.empty(M, N1, dtype=torch.float16, device="cuda")
        C2 = torch.empty(M, N2, dtype=torch.float16, device="cuda")
        torch.cuda.synchronize()
        for sched in (pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC, pts.GEMM_SCHED_NONPERSISTENT):
            with torch.cuda.stream(s):
                C1.fill_(float("nan"))
                C2.fill_(float("nan"))
            pts.gemm_run(h, M, N1, K1, A1, B1, C1, wl.F16, sched, 1.0, 1.0, s)
            pts.gemm_run(h, M, N2, N1, C1, B2, C2, wl.F16, sched, 1.0, 1.0, s)
            assert pts.gemm_check(h, s)[0] == 0
            x2 = wl.Inputs(wl.Problem("chain", M, N2, N1, wl.F16, "uniform", 0), C1.cpu(), b2.A, 1.0, 1.0)
            assert compare_full(x2, C2, what="chain, second GEMM") <= TOL[wl.F16]
            assert compare_full(x1, C1, what="chain, first GEMM") <= TOL[wl.F16]
    finally:
        pts.gemm_destroy(h)
