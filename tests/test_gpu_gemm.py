"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Element by element on small and ragged shapes (several tiles plus partial
tiles), on sampled outputs at the full workload sizes, bit-exact on closed
forms, and tile coverage bit-exact against the scheduler model.
Tolerance (max relative error normalised by s * sum_k |a||b|): 2e-3 for
fp16/bf16, 3e-2 for e4m3 after per-tensor scaling.
"""
import numpy as np
import pytest
import torch

import persistent_tile_scheduled_gb300 as pts
import workloads as wl
from oracle import gemm as og

from helpers import (TOL, check_records, compare_full, compare_sampled, run_device)

pytestmark = pytest.mark.gpu

SCHEDS = [pts.GEMM_SCHED_NONPERSISTENT, pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC]


# the wide tile (128 x 256 per CTA) with single CTAs and with CTA pairs, the
# narrow tile (128 x 128 per CTA, two CTAs per SM) and its pair form (256 x 128
# per CTA pair, one CTA per SM)
SHAPES = {"cg1": dict(cta_group=1), "cg2": dict(cta_group=2), "narrow": dict(cta_group=1, tile_n=128),
          "narrow_cg2": dict(cta_group=2, tile_n=128)}


@pytest.fixture(scope="module", params=list(SHAPES), ids=list(SHAPES))
def handle(request):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS, **SHAPES[request.param]))
    yield h, request.param
    pts.gemm_destroy(h)


def _run_checked(h, x, sched, full=True):
    p = x.problem
    C = run_device(h, x, sched)
    info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, sched)
    st, recs, dev = pts.gemm_read_debug(h, int(info.work_items))
    assert st == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
    check_records(recs, info, sched, p.K)
    err = compare_full(x, C) if full else compare_sampled(x, C, info.tile_m, info.tile_n)
    assert err <= TOL[p.dtype], f"rel err {err}"
    return C, err


@pytest.mark.parametrize("sched", SCHEDS)
def test_fp16_512_all_schedulers(handle, sched):
    h, _ = handle
    x = wl.make_inputs(wl.fp16_512()[0])
    _run_checked(h, x, sched)


RAGGED = [(1, 8, 16), (129, 264, 80), (300, 520, 208), (257, 8, 16), (640, 1000, 1040), (2000, 48, 64)]


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16, wl.E4M3])
@pytest.mark.parametrize("shape", RAGGED, ids=[f"{m}x{n}x{k}" for m, n, k in RAGGED])
@pytest.mark.parametrize("sched", SCHEDS)
def test_ragged_shapes(handle, dtype, shape, sched):
    h, _ = handle
    M, N, K = shape
    dist = "normal" if dtype == wl.E4M3 else "uniform"
    x = wl.make_inputs(wl.Problem("ragged", M, N, K, dtype, dist, 17 + M + N + K))
    _run_checked(h, x, sched)


@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16, wl.E4M3])
def test_identity_and_permutation_bit_exact(handle, dtype):
    """One non-zero product per output: the result is exactly b (or permuted b)."""
    h, _ = handle
    M = K = 512
    N = 264
    rng = np.random.default_rng(5)
    perm = rng.permutation(K)
    P = np.zeros((M, K), np.float32)
    P[np.arange(M), perm] = 1.0
    td = {wl.F16: torch.float16, wl.BF16: torch.bfloat16, wl.E4M3: torch.float8_e4m3fn}[dtype]
    Bv = torch.from_numpy(rng.uniform(-2, 2, (N, K)).astype(np.float32)).to(td)
    for mat in (np.eye(M, dtype=np.float32), P):
        A = torch.from_numpy(mat).to(td)
        x = wl.Inputs(wl.Problem("perm", M, N, K, dtype, "uniform", 0), A, Bv, 1.0, 1.0)
        C = run_device(h, x, pts.GEMM_SCHED_CLC)
        st, dev = pts.gemm_check(h)
        assert st == 0
        b = Bv.double().numpy().T                           # K x N
        want = b[np.nonzero(mat)[1], :]
        got = C.double().cpu().numpy()
        assert np.array_equal(got, want)


def test_k_zero_writes_zeros(handle):
    h, _ = handle
    C = torch.full((64, 48), 7.0, dtype=torch.float16, device="cuda")
    pts.gemm_run(h, 64, 48, 0, None, None, C, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
    torch.cuda.synchronize()
    assert not C.any()


def test_empty_m_or_n_launches_nothing(handle):
    h, _ = handle
    pts.gemm_run(h, 0, 64, 64, None, None, None, pts.GEMM_BF16, pts.GEMM_SCHED_CLC)
    pts.gemm_run(h, 64, 0, 64, None, None, None, pts.GEMM_BF16, pts.GEMM_SCHED_CLC)
    assert pts.gemm_check(h)[0] == 0


def test_invalid_arguments_are_rejected(handle):
    h, _ = handle
    A = torch.zeros(64, 72, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(pts.GemmError):     # K not a multiple of 8
        pts.gemm_run(h, 64, 64, 12, A, A, C, pts.GEMM_F16, 1)
    with pytest.raises(pts.GemmError):     # misaligned pointer
        pts.gemm_run(h, 64, 64, 64, A.data_ptr() + 2, A, C, pts.GEMM_F16, 1)
    with pytest.raises(pts.GemmError):     # bad scheduler
        pts.gemm_run(h, 64, 64, 64, A, A, C, pts.GEMM_F16, 7)
    with pytest.raises(pts.GemmError):     # e4m3 scale must be positive
        pts.gemm_run(h, 64, 64, 64, A, A, C, pts.GEMM_E4M3, 1, 0.0, 1.0)


def test_run_host_matches_device_path(handle):
    h, _ = handle
    x = wl.custom(300, 264, 128, wl.BF16, "uniform", 3)
    Cd = run_device(h, x, pts.GEMM_SCHED_STATIC)
    Ch = torch.empty(300, 264, dtype=torch.bfloat16).pin_memory()
    pts.gemm_run_host(h, 300, 264, 128, x.A.pin_memory(), x.B.pin_memory(), Ch, wl.BF16, pts.GEMM_SCHED_STATIC)
    assert torch.equal(Cd.cpu().view(torch.int16), Ch.view(torch.int16))


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("sched", SCHEDS)
def test_forced_column_slices(cg, split, sched):
    """Every tile cut into 2 or 4 column slices (MMA N = 128 or 64), ragged shapes."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, split=split, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1040, wl.F16), (257, 264, 96, wl.E4M3)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("slices", M, N, K, dt, dist, M + N + K + split))
            _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("G", [3, 5])
@pytest.mark.parametrize("sched", SCHEDS)
def test_forced_stream_k_share(cg, G, sched):
    """The last waves shared stream-K style on G clusters: each unit's k-block
    range cut at tile boundaries into pieces; a tile split between two units
    is summed by the fixup (the first piece to finish writes its fp32 partial,
    the other adds it and stores C).  Ragged shapes, every dtype."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, split_k=1, max_clusters=G,
                                         debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1040, wl.F16), (257, 264, 512, wl.E4M3),
                              (1000, 1800, 2000, wl.BF16)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("streamk", M, N, K, dt, dist, M + N + K + 10 * G))
            info = pts.gemm_query(h, M, N, K, dt, sched)
            T = int(info.tiles)
            assert info.split_k == (1 if T >= G and T % G else 0)
            if info.split_k:
                assert (info.sk_tiles, info.sk_units) == (T % G + G, G)
                assert info.work_items == 3 * G + T - info.sk_tiles and info.units == G + T - info.sk_tiles
            for _ in range(2):      # twice: the claim counters of one launch must not leak into the next
                _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("G", [3, 5])
@pytest.mark.parametrize("sched", SCHEDS)
def test_tail_halves(cg, G, sched):
    """A partial last wave of R <= G/2 tiles on G clusters: under the
    persistent schedulers those tiles run as two column halves each, so every
    cluster busy in the last wave holds half a tile (the non-persistent grid
    keeps whole tiles).  Records bit-exact against the scheduler model, parity against the
    oracle, and the same bits as with whole tiles (split 1, no stream-K
    share): a half changes which cluster computes a column, not its sum.
    Ragged shapes, every dtype."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, max_clusters=G, debug_flags=pts.GEMM_DEBUG_RECORDS))
    h1 = pts.gemm_create(0, pts.make_opts(cta_group=cg, max_clusters=G, split=1, split_k=-1))
    tails = 0
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1040, wl.F16), (257, 264, 512, wl.E4M3),
                              (1000, 1800, 2000, wl.BF16), (1100, 1304, 640, wl.F16)]:
            info = pts.gemm_query(h, M, N, K, dt, sched)
            T = int(info.tiles)
            R = T % G
            want = R if (sched != pts.GEMM_SCHED_NONPERSISTENT and T > G and 0 < 2 * R <= G) else 0
            assert int(info.tail_tiles) == want, (M, N, K)
            assert info.split_k == 0 or not want, (M, N, K)   # the halves replace the share
            if want:
                assert info.units == T + R and info.work_items == T + R and info.split == 1
                assert int(pts.gemm_query(h1, M, N, K, dt, sched).tail_tiles) == 0
            tails += want > 0
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("tail", M, N, K, dt, dist, M + N + K + 10 * G))
            C, _ = _run_checked(h, x, sched)
            if info.split_k == 0:   # (the share's fixup sums in another order)
                C1 = run_device(h1, x, sched)
                assert pts.gemm_check(h1)[0] == 0
                assert torch.equal(C, C1), (M, N, K)
    finally:
        pts.gemm_destroy(h)
        pts.gemm_destroy(h1)
    assert tails > 0 or sched == pts.GEMM_SCHED_NONPERSISTENT


@pytest.mark.parametrize("cg,stages", [(1, 2), (1, 3), (1, 4), (2, 2), (2, 3)])
def test_every_ring_depth(cg, stages):
    """Shallower rings than the default: a single CTA's stage holds one k-block,
    a pair's two (so an item with an odd k-block count ends on a half stage)."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, stages=stages, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        assert pts.gemm_query(h, 512, 512, 512, pts.GEMM_F16, 1).stages == stages
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1088, wl.F16), (257, 264, 384, wl.E4M3)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("ring", M, N, K, dt, dist, M + N + K + stages))
            for sched in SCHEDS:
                _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("split,split_k,G", [(1, -1, 0), (2, 0, 0), (1, 1, 5), (0, 0, 5)])
def test_direct_store_epilogue(cg, split, split_k, G):
    """The epilogue that stores C rows straight from registers (no TMA store):
    whole tiles, column slices, stream-K pieces, and the library's own plan on
    5 clusters (tail halves where the last wave leaves at most 2 tiles)."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=cg, epilogue=2, split=split, split_k=split_k, max_clusters=G,
                                         debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1040, wl.F16), (257, 264, 512, wl.E4M3)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("direct", M, N, K, dt, dist, M + N + K + 3))
            for sched in SCHEDS:
                _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


def test_automatic_stream_k_share():
    """A partial last wave is shared stream-K style when that saves time."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=2, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        info = pts.gemm_query(h, 4096, 4096, 8192, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
        G, T = int(info.max_active_clusters), int(info.tiles)
        if T % G:
            assert info.split_k == 1 and (info.sk_tiles, info.sk_units) == (T % G + G, G)
        h1 = pts.gemm_create(0, pts.make_opts(cta_group=1))
        try:
            G1 = int(pts.gemm_query(h1, 4096, 4096, 128, pts.GEMM_F16, 1).max_active_clusters)
            info = pts.gemm_query(h1, 4096, 4096, 128, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
            assert info.split_k == 0 and info.sk_tiles == 0   # 2 k-blocks: saves less than the fixup costs
            info = pts.gemm_query(h1, 128 * G1, 256, 4096, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
            assert info.split_k == 0                    # whole waves: nothing to share
        finally:
            pts.gemm_destroy(h1)
        x = wl.make_inputs(wl.Problem("k8192", 4096, 4096, 8192, wl.F16, "normal_sqrtk", 77))
        for sched in SCHEDS:
            _run_checked(h, x, sched, full=False)
    finally:
        pts.gemm_destroy(h)


def test_automatic_cta_group():
    """CTA pairs from 14 k-blocks per tile for the persistent schedulers, from
    64 for the non-persistent grid; single CTAs below."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=0))
    try:
        assert pts.gemm_query(h, 4096, 4096, 512, pts.GEMM_F16, 1).cta_group == 1      # 8 k-blocks
        assert pts.gemm_query(h, 4096, 4096, 832, pts.GEMM_F16, 1).cta_group == 1      # 13
        assert pts.gemm_query(h, 4096, 4096, 840, pts.GEMM_F16, 1).cta_group == 2      # 14 (a partial one)
        assert pts.gemm_query(h, 4096, 4096, 8192, pts.GEMM_BF16, 1).cta_group == 2    # 128
        assert pts.gemm_query(h, 8192, 8192, 1664, pts.GEMM_E4M3, 1).cta_group == 1    # 13 (128-wide k-blocks)
        assert pts.gemm_query(h, 8192, 8192, 1792, pts.GEMM_E4M3, 1).cta_group == 2    # 14
        assert pts.gemm_query(h, 4096, 4096, 840, pts.GEMM_F16, 2).cta_group == 2      # CLC as static
        NP = pts.GEMM_SCHED_NONPERSISTENT
        assert pts.gemm_query(h, 4096, 4096, 1024, pts.GEMM_F16, NP).cta_group == 1    # 16
        assert pts.gemm_query(h, 4096, 4096, 4032, pts.GEMM_F16, NP).cta_group == 1    # 63
        assert pts.gemm_query(h, 4096, 4096, 4096, pts.GEMM_F16, NP).cta_group == 2    # 64
        assert pts.gemm_query(h, 8192, 8192, 8192, pts.GEMM_BF16, NP).cta_group == 2   # 128
        x1 = wl.custom(640, 1000, 2048, wl.F16, "normal_sqrtk", 13)                   # 32: single CTAs
        C1 = run_device(h, x1, NP)
        assert pts.gemm_check(h)[0] == 0
        assert compare_full(x1, C1) <= TOL[wl.F16]
        x = wl.custom(640, 1000, 8192, wl.BF16, "normal_sqrtk", 12)
        C = run_device(h, x, pts.GEMM_SCHED_CLC)
        assert pts.gemm_check(h)[0] == 0
        assert compare_full(x, C) <= TOL[wl.BF16]
    finally:
        pts.gemm_destroy(h)


def test_automatic_slicing_of_sub_wave_problems():
    """Problems smaller than a wave are sliced so that more SMs take part."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=1))
    try:
        info = pts.gemm_query(h, 4096, 4096, 4096, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
        assert info.split == 1                              # past one wave: never column slices
        info = pts.gemm_query(h, 512, 512, 512, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
        assert info.tiles == 8 and info.split == 4 and info.sk_tiles == 0 and info.work_items == 32
    finally:
        pts.gemm_destroy(h)


def test_many_buffer_sets_on_one_handle():
    """More distinct A, B, C buffers than the tensor-map cache has slots, with
    every cut of the tiles in play: maps evicted from the cache, even within
    one call, never leak into a launch."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=2, timeout_ns=200_000_000))
    try:
        shapes = [(4096, 4096, k) for k in range(2816, 4097, 128)] + [(512, 512, 512), (384, 264, 1024)]
        outs = []
        for i, (M, N, K) in enumerate(shapes * 2):
            x = wl.custom(M, N, K, wl.F16, "normal_sqrtk", 900 + i)
            outs.append((x, run_device(h, x, pts.GEMM_SCHED_STATIC)))
        st, dev = pts.gemm_check(h)
        assert st == 0, f"device word {dev:#x}"
        for x, C in outs[-4:]:
            p = x.problem
            assert compare_sampled(x, C, 256, 256) <= TOL[wl.F16]
    finally:
        pts.gemm_destroy(h)


def test_run_host_batch_matches_device_path(handle):
    """Overlapped host-buffer batch: every result equals the device-path result."""
    h, _ = handle
    xs = [wl.custom(300, 264, 128, wl.BF16, "uniform", 31), wl.custom(1000, 520, 1024, wl.F16, "uniform", 32),
          wl.custom(640, 1000, 256, wl.E4M3, "normal", 33), wl.custom(8, 8, 16, wl.BF16, "uniform", 34),
          wl.custom(513, 256, 64, wl.F16, "uniform", 35)]
    want, batch = [], []
    for x in xs:
        p = x.problem
        want.append(run_device(h, x, pts.GEMM_SCHED_CLC).cpu())
        C = torch.empty(p.M, p.N, dtype=wl.output_torch_dtype(p.dtype)).pin_memory()
        batch.append((p.M, p.N, p.K, x.A.pin_memory(), x.B.pin_memory(), C, p.dtype, x.scale_a, x.scale_b))
    pts.gemm_run_host_batch(h, batch, pts.GEMM_SCHED_CLC)
    for w, q in zip(want, batch):
        assert torch.equal(w.view(torch.int16), q[5].view(torch.int16))


# ------------------------------------------------- the common launch's kernel

COMMON = [(300, 520, 208), (640, 1000, 1040), (2000, 48, 64), (1000, 1800, 2000), (1, 8, 16)]


@pytest.mark.parametrize("shape_name", list(SHAPES))
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16, wl.E4M3])
@pytest.mark.parametrize("sched", SCHEDS)
def test_common_launch_kernel_matches_the_full_one(shape_name, dtype, sched):
    """A launch that needs none of the debug and extra features runs a kernel
    built with them compiled out.  It must give the same bits as the full
    kernel (selected here by asking for debug records) on every tile shape,
    dtype and scheduler -- ragged shapes, column slices, the stream-K share --
    and match the oracle."""
    kw = SHAPES[shape_name]
    h_common = pts.gemm_create(0, pts.make_opts(**kw))
    h_full = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS, **kw))
    try:
        for M, N, K in COMMON:
            if dtype == wl.E4M3:
                K = (K + 15) // 16 * 16
            dist = "normal" if dtype == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("common", M, N, K, dtype, dist, 31 + M + N + K))
            C0 = run_device(h_common, x, sched)
            assert pts.gemm_check(h_common)[0] == 0
            C1 = run_device(h_full, x, sched)
            assert pts.gemm_check(h_full)[0] == 0
            assert torch.equal(C0.view(torch.int16), C1.view(torch.int16)), (shape_name, M, N, K)
            assert compare_full(x, C0, what="common-launch kernel") <= TOL[dtype]
    finally:
        pts.gemm_destroy(h_common)
        pts.gemm_destroy(h_full)


@pytest.mark.slow
@pytest.mark.parametrize("name,arg", [("fp16_4096_ksweep", 128), ("fp16_4096_ksweep", 1024),
                                      ("fp16_4096_ksweep", 4096), ("bf16_8192_ksweep", 8192), ("e4m3_8192", None)],
                         ids=["fp16-K128", "fp16-K1024", "fp16-K4096", "bf16-8192", "e4m3-8192"])
def test_common_launch_kernel_at_full_size(name, arg):
    """The workloads bench.py times, with the library's defaults: the common
    launch's kernel gives the bits of the full kernel under every scheduler,
    and matches the oracle on a sample."""
    h_common = pts.gemm_create(0, pts.make_opts())
    h_full = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        x = wl.make_inputs(_full_problem(name, arg))
        p = x.problem
        for sched in SCHEDS:
            C0 = run_device(h_common, x, sched)
            assert pts.gemm_check(h_common)[0] == 0
            C1 = run_device(h_full, x, sched)
            assert pts.gemm_check(h_full)[0] == 0
            assert torch.equal(C0.view(torch.int16), C1.view(torch.int16)), (name, arg, sched)
            info = pts.gemm_query(h_common, p.M, p.N, p.K, p.dtype, sched)
            assert compare_sampled(x, C0, info.tile_m, info.tile_n, what="common-launch kernel") <= TOL[p.dtype]
    finally:
        pts.gemm_destroy(h_common)
        pts.gemm_destroy(h_full)


# ------------------------------------------------------------- narrow tile

def test_narrow_tile_keeps_two_ctas_per_sm():
    """The narrow tile's ring, staging and accumulators fit twice per SM: the
    static grid holds two CTAs per SM (twice as many programs as SMs)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    h = pts.gemm_create(0, pts.make_opts(tile_n=128))
    try:
        for dt, K in ((wl.F16, 512), (wl.BF16, 256), (wl.E4M3, 1024)):
            info = pts.gemm_query(h, 4096, 4096, K, dt, pts.GEMM_SCHED_STATIC)
            assert (info.tile_m, info.tile_n, info.cta_group, info.ctas_per_sm) == (128, 128, 1, 2)
            assert info.max_active_clusters == 2 * sms
            assert info.grid_ctas == 2 * sms and info.tiles == 32 * 32 and info.split_k == 0
            assert info.smem_bytes * 2 <= 228 * 1024
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("sched", [pts.GEMM_SCHED_NONPERSISTENT, pts.GEMM_SCHED_CLC])
def test_narrow_tile_runs_two_ctas_on_one_sm(sched):
    """The hardware does co-schedule two narrow-tile CTAs per SM: in a launch
    of one CTA per tile, the per-item records (SM id, MMA start and last store
    times) show two CTAs active at once on every SM, and never three."""
    h = pts.gemm_create(0, pts.make_opts(tile_n=128, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        x = wl.make_inputs(wl.fp16_4096_ksweep([512])[0])
        p = x.problem
        _run_checked(h, x, sched, full=False)
        info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, sched)
        run_device(h, x, sched)
        st, recs, dev = pts.gemm_read_debug(h, int(info.work_items))
        assert st == 0
        ref = recs[0].t_mma_start

        def rel(t):   # the records keep the low 32 bits of %globaltimer (ns)
            return ((t - ref + (1 << 31)) & 0xFFFFFFFF) - (1 << 31)

        spans = {}
        for i in range(int(info.work_items)):
            r = recs[i]
            sm, t0, t1 = spans.get(r.owner, (r.smid, 1 << 40, -(1 << 40)))
            spans[r.owner] = (sm, min(t0, rel(r.t_mma_start)), max(t1, rel(r.t_stored)))
        per_sm = {}
        for sm, t0, t1 in spans.values():
            per_sm.setdefault(sm, []).append((t0, t1))
        most = {}
        for sm, iv in per_sm.items():
            events = sorted([(t0, 1) for t0, _ in iv] + [(t1, -1) for _, t1 in iv], key=lambda e: (e[0], e[1]))
            c = m = 0
            for _, d in events:
                c += d
                m = max(m, c)
            most[sm] = m
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert len(most) == sms
        assert max(most.values()) == 2
        assert sum(1 for m in most.values() if m == 2) >= sms * 3 // 4, most
    finally:
        pts.gemm_destroy(h)


def test_automatic_tile_choice():
    """With the shape left to the library, the non-persistent grid takes the
    narrow tile for tiles of at most 4 k-blocks; the persistent grids, and a
    caller that fixes the CTA group, get the wide tile."""
    h = pts.gemm_create(0, pts.make_opts())
    h1 = pts.gemm_create(0, pts.make_opts(cta_group=1))
    try:
        for dt, K, narrow in ((wl.F16, 128, True), (wl.F16, 256, True), (wl.F16, 320, False),
                              (wl.E4M3, 512, True), (wl.E4M3, 640, False), (wl.BF16, 4096, False)):
            info = pts.gemm_query(h, 4096, 4096, K, dt, pts.GEMM_SCHED_NONPERSISTENT)
            assert info.tile_n == (128 if narrow else 256), (dt, K)
            for sched in (pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC):
                assert pts.gemm_query(h, 4096, 4096, K, dt, sched).tile_n == 256
            for sched in SCHEDS:
                assert pts.gemm_query(h1, 4096, 4096, K, dt, sched).tile_n == 256
    finally:
        pts.gemm_destroy(h)
        pts.gemm_destroy(h1)


def test_narrow_tile_rejects_what_it_lacks():
    for bad in (dict(tile_n=128, split=4), dict(tile_n=128, split_k=1), dict(tile_n=128, cta_group=2, split=4),
                dict(tile_n=64)):
        with pytest.raises(pts.GemmError):
            pts.gemm_create(0, pts.make_opts(**bad))


def test_narrow_pair_tile_shape():
    """The narrow tile's pair form: 256 x 128 per CTA pair, one CTA per SM, a
    ring of four two-k-block stages, so the static grid holds one pair per two
    SMs; never chosen by the library on its own."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    h = pts.gemm_create(0, pts.make_opts(tile_n=128, cta_group=2))
    h0 = pts.gemm_create(0, pts.make_opts())
    try:
        for dt, K in ((wl.F16, 512), (wl.BF16, 4096), (wl.E4M3, 1024)):
            info = pts.gemm_query(h, 4096, 4096, K, dt, pts.GEMM_SCHED_STATIC)
            assert (info.tile_m, info.tile_n, info.cta_group, info.ctas_per_sm) == (256, 128, 2, 1)
            assert info.stages == 4 and info.max_active_clusters == sms // 2
            assert info.grid_ctas == sms and info.tiles == 16 * 32 and info.split_k == 0
            for sched in SCHEDS:
                auto = pts.gemm_query(h0, 4096, 4096, K, dt, sched)
                assert not (auto.tile_n == 128 and auto.cta_group == 2)
        # below one wave: column halves at most
        assert pts.gemm_query(h, 300, 520, 208, wl.BF16, pts.GEMM_SCHED_STATIC).split == 2
    finally:
        pts.gemm_destroy(h)
        pts.gemm_destroy(h0)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("sched", SCHEDS)
def test_narrow_tile_column_halves(sched, cg):
    """Sub-wave problems on the narrow tile (and its pair form) are cut into
    64-column halves."""
    h = pts.gemm_create(0, pts.make_opts(tile_n=128, cta_group=cg, split=2, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (640, 1000, 1040, wl.F16), (257, 264, 96, wl.E4M3)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("narrow", M, N, K, dt, dist, M + N + K + 2))
            info = pts.gemm_query(h, M, N, K, dt, sched)
            assert info.split == 2 and info.tile_n == 128
            _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("K", [128, 256, 512])
def test_narrow_tile_sweep_points_sampled(K):
    """The fp16 4096 sweep's small-K end on the narrow tile, two CTAs per SM,
    every scheduler (the library's plan for the non-persistent grid at K =
    128 and 256)."""
    h = pts.gemm_create(0, pts.make_opts(tile_n=128, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        x = wl.make_inputs(wl.fp16_4096_ksweep([K])[0])
        for sched in SCHEDS:
            info = pts.gemm_query(h, 4096, 4096, K, wl.F16, sched)
            assert info.tile_n == 128 and info.ctas_per_sm == 2
            _run_checked(h, x, sched, full=False)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("K", [512, 4096])
def test_narrow_pair_tile_sweep_points_sampled(K):
    """Full-size fp16 4096^2 points on the narrow tile's pair form (512 tiles
    of 256 x 128 on 76 pairs), every scheduler, every work item's record
    checked against the scheduler model."""
    h = pts.gemm_create(0, pts.make_opts(tile_n=128, cta_group=2, debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        x = wl.make_inputs(wl.fp16_4096_ksweep([K])[0])
        for sched in SCHEDS:
            info = pts.gemm_query(h, 4096, 4096, K, wl.F16, sched)
            assert (info.tile_m, info.tile_n, info.cta_group) == (256, 128, 2)
            _run_checked(h, x, sched, full=False)
    finally:
        pts.gemm_destroy(h)


# ------------------------------------------------------- long and skinny

LONG = [(300, 264, 65536, wl.BF16), (1, 8, 8192, wl.F16), (8, 4096, 4096, wl.BF16), (4096, 8, 2048, wl.E4M3),
        (129, 1032, 24576, wl.F16)]


@pytest.mark.slow
@pytest.mark.parametrize("shape", LONG, ids=[f"{m}x{n}x{k}-{wl.DTYPE_NAMES[d]}" for m, n, k, d in LONG])
def test_long_and_skinny_problems(shape):
    """Library defaults on long accumulations (up to 1024 k-blocks per tile,
    column slices below one wave) and on single-row, single-tile-column and
    eight-column outputs, every scheduler, element by element."""
    M, N, K, dt = shape
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        dist = "normal" if dt == wl.E4M3 else "normal_sqrtk"
        x = wl.make_inputs(wl.Problem("long", M, N, K, dt, dist, M + N + K))
        for sched in SCHEDS:
            _run_checked(h, x, sched)
    finally:
        pts.gemm_destroy(h)


MANY = [(262144, 24, 64, wl.BF16), (16, 131072, 64, wl.F16), (65536, 40, 128, wl.E4M3)]


@pytest.mark.slow
@pytest.mark.parametrize("shape", MANY, ids=[f"{m}x{n}x{k}-{wl.DTYPE_NAMES[d]}" for m, n, k, d in MANY])
@pytest.mark.parametrize("sched", SCHEDS)
def test_many_tiles_along_one_dimension(handle, shape, sched):
    """Thousands of tiles along M (one tile column) or hundreds to a thousand
    along N (one tile row): the grouped order crosses hundreds of group
    boundaries or keeps one short group, non-persistent grids of thousands of
    clusters, static strides over many waves.  Every work item's record is
    checked against the scheduler model; outputs on a sample."""
    h, _ = handle
    M, N, K, dt = shape
    dist = "normal" if dt == wl.E4M3 else "normal_sqrtk"
    x = wl.make_inputs(wl.Problem("many", M, N, K, dt, dist, M + 3 * N + K))
    _run_checked(h, x, sched, full=False)


# ---------------------------------------------------------------- full sizes

FULL = ([("fp16_4096_ksweep", k) for k in (128, 2048, 4096)]
        + [("bf16_8192_ksweep", k) for k in (256, 8192)]
        + [("e4m3_8192", None), ("e4m3_8192_k", 2048)]
        + [("bf16_tail", i) for i in range(3)])


def _full_problem(name, arg):
    if name == "fp16_4096_ksweep":
        return wl.fp16_4096_ksweep([arg])[0]
    if name == "bf16_8192_ksweep":
        return wl.bf16_8192_ksweep([arg])[0]
    if name == "e4m3_8192":
        return wl.e4m3_8192()[0]
    if name == "e4m3_8192_k":   # e4m3 at a K whose last wave runs as column halves
        return wl.Problem(f"e4m3_8192_k{arg}", 8192, 8192, arg, wl.E4M3, "normal", 4000 + arg)
    return wl.bf16_tail()[arg]


@pytest.mark.slow
@pytest.mark.parametrize("name,arg", FULL, ids=[f"{n}-{a}" for n, a in FULL])
def test_full_size_sampled(handle, name, arg):
    h, _ = handle
    x = wl.make_inputs(_full_problem(name, arg))
    for sched in SCHEDS:
        _run_checked(h, x, sched, full=False)


@pytest.mark.slow
@pytest.mark.parametrize("K", [128, 1024, 1792, 2560, 3072, 4096])
def test_bench_configuration_sampled(K):
    """The exact launch configuration bench.py times: library defaults (CTA
    group, ring depth, last-wave plan chosen per GEMM) on sweep GEMMs that take
    each plan: single CTAs and CTA pairs with the last wave's tiles in column
    halves, and CTA pairs with the stream-K share."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS))
    try:
        x = wl.make_inputs(wl.fp16_4096_ksweep([K])[0])
        info = pts.gemm_query(h, 4096, 4096, K, pts.GEMM_F16, pts.GEMM_SCHED_STATIC)
        assert info.cta_group == (2 if K // 64 >= 14 else 1)
        assert (info.split_k, int(info.tail_tiles) > 0) == ((1, False) if K // 64 >= 48 else (0, True))
        for sched in SCHEDS:
            _run_checked(h, x, sched, full=False)
    finally:
        pts.gemm_destroy(h)


# ---------------------------------------------------------------- CLC extras

@pytest.mark.parametrize("stop_at", [0, 1, 3])
def test_clc_injected_request_failure_keeps_coverage(stop_at):
    """Every CTA behaves as if its stop_at-th request had failed; the clusters
    it would have cancelled launch and run their own tiles."""
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS | pts.GEMM_DEBUG_CLC_STOP_AT,
                                         fault_arg=stop_at))
    try:
        x = wl.custom(2048, 2048, 256, wl.BF16, "uniform", 11)
        _run_checked(h, x, pts.GEMM_SCHED_CLC)
        x = wl.custom(4096, 4096, 256, wl.BF16, "uniform", 12)   # several waves, the last in column halves
        assert pts.gemm_query(h, 4096, 4096, 256, wl.BF16, pts.GEMM_SCHED_CLC).tail_tiles > 0
        _run_checked(h, x, pts.GEMM_SCHED_CLC, full=False)
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("stop_at", [None, 0, 2])
def test_clc_claiming_two_units_ahead(shape, stop_at):
    """clc_depth 2: a cluster claims its next unit one unit earlier than with
    depth 1 (still one request at a time).  Coverage stays exact, with and
    without a request that behaves as failed, on ragged and multi-wave
    problems, stream-K units and tail halves included."""
    flags = pts.GEMM_DEBUG_RECORDS | (pts.GEMM_DEBUG_CLC_STOP_AT if stop_at is not None else 0)
    h = pts.gemm_create(0, pts.make_opts(clc_depth=2, debug_flags=flags, fault_arg=stop_at or 0, **SHAPES[shape]))
    try:
        for (M, N, K, dt) in [(300, 520, 208, wl.BF16), (2048, 2048, 256, wl.F16), (1000, 1800, 2000, wl.BF16),
                              (640, 1000, 512, wl.E4M3), (4096, 4096, 256, wl.F16)]:
            dist = "normal" if dt == wl.E4M3 else "uniform"
            x = wl.make_inputs(wl.Problem("clc2", M, N, K, dt, dist, M + N + K + 5))
            _run_checked(h, x, pts.GEMM_SCHED_CLC, full=M < 4096)
    finally:
        pts.gemm_destroy(h)


def test_clc_depth_option_is_checked():
    for bad in (-1, 3):
        with pytest.raises(pts.GemmError):
            pts.gemm_create(0, pts.make_opts(clc_depth=bad))


def test_two_gemms_on_two_streams():
    """Two CLC GEMMs in flight at once on one GPU: both exact in coverage and
    within tolerance (the concurrency case CLC redistributes work for)."""
    hs = [pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_RECORDS)) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    try:
        xs = [wl.make_inputs(wl.bf16_tail()[0]), wl.make_inputs(wl.bf16_tail()[2])]
        dev_in = [(x.A.cuda(), x.B.cuda()) for x in xs]
        Cs = [torch.empty(x.problem.M, x.problem.N, dtype=torch.bfloat16, device="cuda") for x in xs]
        torch.cuda.synchronize()
        for h, s, x, (A, B), C in zip(hs, streams, xs, dev_in, Cs):
            p = x.problem
            pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_CLC, 1.0, 1.0, s)
        for h, s, x, C in zip(hs, streams, xs, Cs):
            p = x.problem
            info = pts.gemm_query(h, p.M, p.N, p.K, p.dtype, pts.GEMM_SCHED_CLC)
            st, recs, dev = pts.gemm_read_debug(h, int(info.work_items), s)
            assert st == 0
            check_records(recs, info, pts.GEMM_SCHED_CLC, p.K)
            assert compare_sampled(x, C, info.tile_m, info.tile_n) <= TOL[p.dtype]
    finally:
        for h in hs:
            pts.gemm_destroy(h)


@pytest.mark.slow
@pytest.mark.parametrize("sched", SCHEDS)
def test_gemm_started_while_another_holds_half_the_sms(sched):
    """A long GEMM (one 128 x 256 tile per CTA on half the SMs) starts first on
    one stream; 5120^2 x 4096 starts on another while it runs.  Part of the
    second grid then finds no free SM: the static grid's later clusters wait
    for the occupier, CLC's resident clusters take their units over, and the
    stream-K pieces of the second GEMM run with part of the grid not yet
    resident (a piece that adds a partial waits only for a piece that has
    already claimed, so is resident).  Coverage exact and both results within
    tolerance."""
    import time
    half = torch.cuda.get_device_properties(0).multi_processor_count // 2
    xo = wl.make_inputs(wl.Problem("occupier", half * 128, 256, 16384, wl.BF16, "normal_sqrtk", 7300))
    xm = wl.make_inputs(wl.Problem("main", 5120, 5120, 4096, wl.BF16, "normal_sqrtk", 7301))
    ho = pts.gemm_create(0, pts.make_opts(cta_group=1, split=1))
    hm = pts.gemm_create(0, pts.make_opts(cta_group=1, debug_flags=pts.GEMM_DEBUG_RECORDS))
    s_occ, s_main = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        po, pm = xo.problem, xm.problem
        info = pts.gemm_query(hm, pm.M, pm.N, pm.K, pm.dtype, sched)
        assert info.split_k == 1   # the stream-K share is part of this plan
        Ao, Bo = xo.A.cuda(), xo.B.cuda()
        Am, Bm = xm.A.cuda(), xm.B.cuda()
        Co = torch.empty(po.M, po.N, dtype=torch.bfloat16, device="cuda")
        Cm = torch.empty(pm.M, pm.N, dtype=torch.bfloat16, device="cuda")
        # one call each first: a handle's first call sets up its kernel and grows
        # its workspace (cudaMalloc may wait for the device), which would keep
        # the two GEMMs from overlapping
        pts.gemm_run(ho, po.M, po.N, po.K, Ao, Bo, Co, po.dtype, pts.GEMM_SCHED_STATIC, 1.0, 1.0, s_occ)
        pts.gemm_run(hm, pm.M, pm.N, pm.K, Am, Bm, Cm, pm.dtype, sched, 1.0, 1.0, s_main)
        torch.cuda.synchronize()

        def waited(recs):
            # the static grid's clusters that found no free SM started only when
            # the occupier (about 0.07 ms) let go of its SMs
            ref = recs[0].t_mma_start
            first = {}
            for i in range(int(info.work_items)):
                r = recs[i]
                if r.visits:
                    t = ((r.t_mma_start - ref + (1 << 31)) & 0xFFFFFFFF) - (1 << 31)   # wrap-safe, ns
                    first[r.owner] = min(first.get(r.owner, t), t)
            return max(first.values()) - min(first.values()) > 20_000

        for attempt in range(3):   # the host's 25 us spin can overrun (the occupier is then done)
            Co.fill_(float("nan"))
            Cm.fill_(float("nan"))
            torch.cuda.synchronize()
            pts.gemm_run(ho, po.M, po.N, po.K, Ao, Bo, Co, po.dtype, pts.GEMM_SCHED_STATIC, 1.0, 1.0, s_occ)
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 25e-6:   # let the occupier's CTAs become resident
                pass
            pts.gemm_run(hm, pm.M, pm.N, pm.K, Am, Bm, Cm, pm.dtype, sched, 1.0, 1.0, s_main)
            torch.cuda.synchronize()
            assert pts.gemm_check(ho, s_occ)[0] == 0
            st, recs, dev = pts.gemm_read_debug(hm, int(info.work_items), s_main)
            assert st == 0, f"{pts.gemm_status_string(st)}, device word {dev:#x}"
            check_records(recs, info, sched, pm.K)
            if sched != pts.GEMM_SCHED_STATIC or waited(recs):
                break
        if sched == pts.GEMM_SCHED_STATIC:
            assert waited(recs), "no cluster waited for the occupier"
        assert compare_sampled(xm, Cm, info.tile_m, info.tile_n, what="under a half-GPU occupier") <= TOL[pm.dtype]
        assert compare_sampled(xo, Co, 128, 256, what="the occupier") <= TOL[po.dtype]
    finally:
        pts.gemm_destroy(ho)
        pts.gemm_destroy(hm)


# ------------------------------------------------------------ bounded waits

@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("sched", [pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC])
def test_wait_time_out_is_reported_and_the_context_survives(shape, sched):
    """A stage load that never arrives makes the MMA warp's bounded wait run
    out: the launch reports GEMM_ERR_TIMEOUT (nothing traps, nothing hangs) and
    the next GEMM on the same context is exact."""
    x = wl.custom(512, 512, 1024, wl.BF16, "uniform", 2)
    h = pts.gemm_create(0, pts.make_opts(debug_flags=pts.GEMM_DEBUG_FAULT_SKIP_TMA, fault_arg=5,
                                         timeout_ns=20_000_000, **SHAPES[shape]))
    try:
        run_device(h, x, sched)
        st, dev = pts.gemm_check(h)
        assert st == pts.gemm.GEMM_ERR_TIMEOUT
        assert dev >> 24 == 1                          # device error code: time-out
        assert (dev >> 16) & 0xFF in (1, 2, 4)        # a stage, MMA or accumulator wait gave up
        assert pts.gemm_check(h)[0] == 0              # the status block was cleared
    finally:
        pts.gemm_destroy(h)
    h = pts.gemm_create(0, pts.make_opts(**SHAPES[shape]))
    try:
        C = run_device(h, x, sched)
        assert pts.gemm_check(h)[0] == 0
        assert compare_full(x, C) <= TOL[wl.BF16]
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("sched", [pts.GEMM_SCHED_STATIC, pts.GEMM_SCHED_CLC])
def test_stream_k_state_is_cleared_after_a_device_error(sched):
    """A stream-K launch that stops on a wait time-out leaves some cut tiles
    claimed by one piece only (1000 x 1800 x 2000 on five clusters: every
    producer withholds its 40th stage, after each unit's first piece of a cut
    tile has claimed and before the piece that shares that tile).
    gemm_check reports the time-out and zeroes the handle's claim counters and
    ready flags, so the next stream-K launch on the same handle, whose cut
    tiles use the same slots and whose producers stay below the withheld
    stage, is exact."""
    h = pts.gemm_create(0, pts.make_opts(cta_group=1, split_k=1, max_clusters=5, timeout_ns=20_000_000,
                                         debug_flags=pts.GEMM_DEBUG_FAULT_SKIP_TMA, fault_arg=40))
    try:
        x1 = wl.custom(1000, 1800, 2000, wl.BF16, "uniform", 81)
        info1 = pts.gemm_query(h, 1000, 1800, 2000, wl.BF16, sched)
        assert info1.split_k == 1 and int(info1.sk_tiles) == 64 % 5 + 5
        run_device(h, x1, sched)
        st, dev = pts.gemm_check(h)
        assert st == pts.gemm.GEMM_ERR_TIMEOUT, f"status {st}, device word {dev:#x}"
        x2 = wl.custom(300, 520, 208, wl.BF16, "uniform", 82)
        info2 = pts.gemm_query(h, 300, 520, 208, wl.BF16, sched)
        assert info2.split_k == 1 and int(info2.sk_tiles) == 9     # every tile in the stream-K region
        for _ in range(2):
            C = run_device(h, x2, sched)
            st, dev = pts.gemm_check(h)
            assert st == 0, f"status {st}, device word {dev:#x}"
            assert compare_full(x2, C) <= TOL[wl.BF16]
    finally:
        pts.gemm_destroy(h)


@pytest.mark.parametrize("dtype,per_clk", [(wl.F16, 8192), (wl.BF16, 8192), (wl.E4M3, 16384)])
@pytest.mark.parametrize("cg", [1, 2])
def test_tensor_peak_probe_pins_the_per_sm_rate(dtype, per_clk, cg):
    """The dense rate the '% of tensor peak' figures assume: 8192 FLOP per SM
    clock for fp16/bf16 and 16384 for e4m3 (measured by an MMA-only loop)."""
    r = pts.gemm_tensor_peak_probe(0, dtype, cg, 20000)
    assert 0.85 * per_clk <= r["flop_per_clk_per_sm"] <= 1.02 * per_clk, r
    assert 0.5 < r["sm_ghz"] < 2.2, r
