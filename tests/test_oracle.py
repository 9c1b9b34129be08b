"""Pins for the CPU oracle: it is checked against things other than itself.

* the bit decoders against the format definitions (hand-written encodings of
  special values) and, exhaustively, against torch's own casts;
* the C triple loop against a separate pure-Python loop (bit-exact: same
  summation order) and against a numpy decode + fp64 matmul;
* hand-worked products stored under tests/golden/;
* closed forms: identity, permutation, rank-1 with small integers (exact);
* the relative-error metric against planted mistakes.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import gemm as og
import workloads as wl


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        g = json.load(f)
    dt = og.DTYPES[g["dtype"]]
    width = np.uint8 if dt == og.E4M3 else np.uint16
    A = np.array([int(x, 16) for x in g["A_rowmajor_MxK_bits"]], dtype=width)
    B = np.array([int(x, 16) for x in g["B_stored_NxK_bits"]], dtype=width)
    return g, dt, A, B


# ----------------------------------------------------------------- decoders

SPECIAL = {
    # IEEE binary16
    (og.F16, 0x3C00): 1.0, (og.F16, 0xC000): -2.0, (og.F16, 0x7BFF): 65504.0,
    (og.F16, 0x0001): 2.0 ** -24, (og.F16, 0x0400): 2.0 ** -14, (og.F16, 0x3555): 0.333251953125,
    (og.F16, 0x8000): -0.0, (og.F16, 0x7C00): float("inf"),
    # bfloat16
    (og.BF16, 0x3F80): 1.0, (og.BF16, 0xBF80): -1.0, (og.BF16, 0x7F7F): 3.3895313892515355e38,
    (og.BF16, 0x0001): 2.0 ** -133, (og.BF16, 0x0080): 2.0 ** -126, (og.BF16, 0x4049): 3.140625,
    # OCP E4M3
    (og.E4M3, 0x7E): 448.0, (og.E4M3, 0xFE): -448.0, (og.E4M3, 0x38): 1.0, (og.E4M3, 0x01): 2.0 ** -9,
    (og.E4M3, 0x08): 2.0 ** -6, (og.E4M3, 0x07): 7 * 2.0 ** -9, (og.E4M3, 0x44): 3.0,
}


@pytest.mark.parametrize("key", sorted(SPECIAL))
def test_decoders_special_values(key):
    dt, bits = key
    want = SPECIAL[key]
    width = np.uint8 if dt == og.E4M3 else np.uint16
    got_c = og.decode_c(np.array([bits], width), dt)[0]
    got_np = og.decode_np(np.array([bits], width), dt)[0]
    got_py = og._py_decode(bits, dt)
    for got in (got_c, got_np, got_py):
        assert got == want and np.signbit(got) == np.signbit(want)


def test_e4m3_nan_patterns():
    for bits in (0x7F, 0xFF):
        assert np.isnan(og.decode_c(np.array([bits], np.uint8), og.E4M3)[0])
        assert np.isnan(og.decode_np(np.array([bits], np.uint8), og.E4M3)[0])


@pytest.mark.parametrize("dt,tdt", [(og.F16, torch.float16), (og.BF16, torch.bfloat16)])
def test_decoders_exhaustive_16bit(dt, tdt):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(tdt).double().numpy()
    for got in (og.decode_np(bits, dt), og.decode_c(bits, dt)):
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), np.nonzero(~same)[0][:8]


def test_decoders_exhaustive_e4m3():
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).double().numpy()
    for got in (og.decode_np(bits, og.E4M3), og.decode_c(bits, og.E4M3),
                np.array([og._py_decode(int(b), og.E4M3) for b in bits])):
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all()


# ------------------------------------------------------------- hand-worked

@pytest.mark.parametrize("name", ["gemm_textbook_f16.json", "gemm_signed_bf16.json",
                                  "gemm_scaled_e4m3.json"])
def test_golden_products(golden_dir, name):
    g, dt, A, B = _golden(golden_dir, name)
    M, N, K, s = g["M"], g["N"], g["K"], g["s"]
    assert list(og.decode_np(A, dt)) == g["A_values"]
    assert list(og.decode_np(B, dt)) == g["B_values"]
    C, Cabs = og.gemm(M, N, K, A, B, dt, s)
    assert C.tolist() == g["C"]
    assert Cabs.tolist() == g["Cabs"]
    assert og.gemm_loops(M, N, K, A, B, dt, s).tolist() == g["C"]
    Cn, Cabsn = og.gemm_numpy(M, N, K, A, B, dt, s)
    assert Cn.tolist() == g["C"] and Cabsn.tolist() == g["Cabs"]


def test_golden_catches_transposed_b(golden_dir):
    """Reading B as K x N row-major instead of N x K gives a different product."""
    g, dt, A, B = _golden(golden_dir, "gemm_signed_bf16.json")
    wrong = B.reshape(g["N"], g["K"]).T.copy().ravel()
    C, _ = og.gemm(g["M"], g["N"], g["K"], A, wrong, dt, g["s"])
    assert C.tolist() != g["C"]


# ---------------------------------------------------------- random parity

def _random_finite_bits(rng, n, dt):
    x = rng.uniform(-3, 3, size=n).astype(np.float32)
    t = torch.from_numpy(x)
    if dt == og.E4M3:
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    td = torch.float16 if dt == og.F16 else torch.bfloat16
    return t.to(td).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dt", [og.F16, og.BF16, og.E4M3])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 7), (3, 2, 8), (7, 8, 16), (8, 7, 3)])
def test_c_loop_equals_python_loop(dt, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 100 + N * 10 + K + dt)
    A = _random_finite_bits(rng, M * K, dt)
    B = _random_finite_bits(rng, N * K, dt)
    s = 0.375 if dt == og.E4M3 else 1.0
    C, _ = og.gemm(M, N, K, A, B, dt, s)
    assert np.array_equal(C, og.gemm_loops(M, N, K, A, B, dt, s))


@pytest.mark.parametrize("dt", [og.F16, og.BF16, og.E4M3])
def test_c_loop_matches_numpy(dt):
    M, N, K = 37, 29, 83
    rng = np.random.default_rng(7 + dt)
    A = _random_finite_bits(rng, M * K, dt)
    B = _random_finite_bits(rng, N * K, dt)
    C, Cabs = og.gemm(M, N, K, A, B, dt, 1.0)
    Cn, Cabsn = og.gemm_numpy(M, N, K, A, B, dt, 1.0)
    assert np.all(np.abs(C - Cn) <= 1e-13 * Cabs)
    assert np.allclose(Cabs, Cabsn, rtol=1e-14, atol=0)


def test_sampled_equals_full():
    M, N, K = 33, 41, 19
    rng = np.random.default_rng(3)
    A = _random_finite_bits(rng, M * K, og.BF16)
    B = _random_finite_bits(rng, N * K, og.BF16)
    C, Cabs = og.gemm(M, N, K, A, B, og.BF16)
    ii = rng.integers(0, M, 200)
    jj = rng.integers(0, N, 200)
    Cs, Cabss = og.gemm_sampled(M, N, K, A, B, og.BF16, ii, jj)
    assert np.array_equal(Cs, C[ii, jj]) and np.array_equal(Cabss, Cabs[ii, jj])


def test_sampled_rejects_out_of_range():
    A = np.zeros(4, np.uint16)
    with pytest.raises(ValueError):
        og.gemm_sampled(2, 2, 2, A, A, og.F16, [0, 2], [0, 0])


def test_multithreaded_equals_single():
    M, N, K = 64, 48, 40
    rng = np.random.default_rng(5)
    A = _random_finite_bits(rng, M * K, og.F16)
    B = _random_finite_bits(rng, N * K, og.F16)
    C1, _ = og.gemm(M, N, K, A, B, og.F16, nthreads=1)
    C4, _ = og.gemm(M, N, K, A, B, og.F16, nthreads=4)
    assert np.array_equal(C1, C4)


# ------------------------------------------------------------ closed forms

def _enc(vals, dt):
    t = torch.tensor(np.asarray(vals, np.float32))
    if dt == og.E4M3:
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().ravel()
    td = torch.float16 if dt == og.F16 else torch.bfloat16
    return t.to(td).view(torch.int16).numpy().view(np.uint16).ravel()


@pytest.mark.parametrize("dt", [og.F16, og.BF16, og.E4M3])
def test_identity(dt):
    """A = I (K = M): C[i,j] = b[i,j] = B[j*K + i], exactly."""
    M = N = K = 24
    rng = np.random.default_rng(11)
    A = _enc(np.eye(M), dt)
    B = _random_finite_bits(rng, N * K, dt)
    C, _ = og.gemm(M, N, K, A, B, dt)
    assert np.array_equal(C, og.decode_np(B, dt).reshape(N, K).T)


@pytest.mark.parametrize("dt", [og.F16, og.BF16, og.E4M3])
def test_permutation(dt):
    """A = P: row i of C is row perm[i] of b (b[k, j] = B[j*K + k])."""
    M = K = 20
    N = 12
    rng = np.random.default_rng(12)
    perm = rng.permutation(K)
    P = np.zeros((M, K))
    P[np.arange(M), perm] = 1.0
    A = _enc(P, dt)
    B = _random_finite_bits(rng, N * K, dt)
    C, _ = og.gemm(M, N, K, A, B, dt)
    b = og.decode_np(B, dt).reshape(N, K).T       # K x N
    assert np.array_equal(C, b[perm, :])


@pytest.mark.parametrize("dt", [og.F16, og.BF16, og.E4M3])
def test_rank_one_small_integers(dt):
    """A[i,k] = u_i x_k, b[k,j] = y_k v_j  =>  C = u_i v_j sum_k x_k y_k, exact."""
    u, x = np.array([1, -2, 3]), np.array([1, 2, -1, 3, 1])
    y, v = np.array([2, -1, 1, 1, 3]), np.array([-1, 2, 1, 4])
    M, K, N = len(u), len(x), len(v)
    A = _enc(np.outer(u, x), dt)
    B = _enc(np.outer(v, y), dt)                       # stored N x K: B[j, k] = v_j y_k
    C, _ = og.gemm(M, N, K, A, B, dt)
    assert np.array_equal(C, np.outer(u, v) * float(np.dot(x, y)))


def test_scale_factor_is_applied_once():
    A = _enc([[2.0, 4.0]], og.E4M3)
    B = _enc([[8.0, 1.0]], og.E4M3)
    C, Cabs = og.gemm(1, 1, 2, A, B, og.E4M3, s=1.0 / (4.0 * 5.0))
    assert C[0, 0] == 20.0 / 20.0 and Cabs[0, 0] == 1.0


def test_k_zero_gives_zero():
    C, Cabs = og.gemm(3, 2, 0, np.zeros(0, np.uint16), np.zeros(0, np.uint16), og.F16)
    assert not C.any() and not Cabs.any()


# ----------------------------------------------------------------- metric

def test_rel_err_planted_mistakes():
    M, N, K = 16, 16, 64
    rng = np.random.default_rng(2)
    A = _random_finite_bits(rng, M * K, og.BF16)
    B = _random_finite_bits(rng, N * K, og.BF16)
    C, Cabs = og.gemm(M, N, K, A, B, og.BF16)
    assert og.rel_err(C, C, Cabs) == 0.0
    # rounding to the output format moves a value by at most u |x| (RNE):
    # not charged when out_u is given, charged (and possibly above 2e-3 for
    # bf16, whose u = 2^-8) when it is not
    for tdt, u in ((torch.bfloat16, 2.0 ** -8), (torch.float16, 2.0 ** -11)):
        Cr = torch.from_numpy(C).to(tdt).double().numpy()
        assert og.rel_err(Cr, C, Cabs, out_u=u) == 0.0
        assert 0.0 < og.rel_err(Cr, C, Cabs) <= u
    # one output-format ulp too many is charged
    Cr = torch.from_numpy(C).to(torch.bfloat16).double().numpy()
    assert og.rel_err(Cr * (1 + 2.0 ** -6), C, Cabs, out_u=2.0 ** -8) > 0.0
    # a dropped k term, a sign flip and a transposed output all fail it
    a = og.decode_np(A, og.BF16).reshape(M, K)
    b = og.decode_np(B, og.BF16).reshape(N, K)
    dropped = a[:, :-1] @ b[:, :-1].T
    assert og.rel_err(dropped, C, Cabs) > 2e-3
    assert og.rel_err(-C, C, Cabs) > 2e-3
    assert og.rel_err(C.T, C, Cabs) > 2e-3


def test_rel_err_zero_normaliser():
    ref = np.zeros((2, 2))
    assert og.rel_err(np.zeros((2, 2)), ref, np.zeros((2, 2))) == 0.0
    bad = np.zeros((2, 2))
    bad[1, 1] = 1e-30
    assert og.rel_err(bad, ref, np.zeros((2, 2))) == float("inf")
    assert og.rel_err(np.full((1,), np.nan), np.ones(1), np.ones(1)) == float("inf")


# ---------------------------------------------------------------- inputs

def test_inputs_are_seeded_and_shaped():
    p = wl.fp16_512()[0]
    x, y = wl.make_inputs(p), wl.make_inputs(p)
    assert torch.equal(x.A.view(torch.int16), y.A.view(torch.int16))
    assert x.A.shape == (512, 512) and x.B.shape == (512, 512)
    a = og.decode_np(x.bits("A"), og.F16)
    assert a.min() >= -1 and a.max() <= 1


def test_e4m3_inputs_hit_max():
    p = wl.Problem("t", 64, 32, 48, wl.E4M3, "normal", 9)
    x = wl.make_inputs(p)
    a = og.decode_np(x.bits("A"), og.E4M3)
    b = og.decode_np(x.bits("B"), og.E4M3)
    assert np.abs(a).max() == 448.0 and np.abs(b).max() == 448.0
    assert np.isfinite(a).all() and np.isfinite(b).all()


def test_grouped_workload_recipe():
    """64 bf16 problems of 1024 x 1024, K log-uniform in [256, 8192] as
    multiples of 8, drawn the same way every time; problem i seeded 6001 + i."""
    ps, qs = wl.bf16_grouped_vark(), wl.bf16_grouped_vark()
    assert ps == qs and len(ps) == 64
    ks = [p.K for p in ps]
    assert all(p.M == 1024 and p.N == 1024 and p.dtype == wl.BF16 and p.dist == "normal_sqrtk" for p in ps)
    assert all(k % 8 == 0 and 256 <= k <= 8192 for k in ks)
    assert [p.seed for p in ps] == list(range(6001, 6065))
    # log-uniform: about as many problems below the geometric midpoint 2^10.5 as above it
    below = sum(k < 2 ** 10.5 for k in ks)
    assert 20 <= below <= 44
    assert max(ks) / min(ks) > 16   # tile costs differ by more than an order of magnitude

