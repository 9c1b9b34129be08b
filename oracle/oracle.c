/*
 * Plain CPU oracle for C = A . B (test infrastructure only).
 *
 * Only the tests, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this library.  It shares no code, header or constant with the CUDA
 * path: it has its own bit decoders and its own loop.  Nothing here is blocked,
 * fused or reordered: each output is the fp64 sum over k in increasing order.
 *
 * What it computes (the plain definition of the GEMM the pages benchmark:
 * "question about persistent kernel concept", the question paragraph, GEMM
 * split into output tiles; "[Persistent] Performance on 09-persistent-matmul on
 * A100 worse than non-persistent", the issue body, the fp16 matmul sweeps):
 *
 *     C[i,j] = s * sum_{k<K} a[i,k] * b[k,j]
 *
 * a[i,k] = value of A[i*K + k]     (A is M x K row-major)
 * b[k,j] = value of B[j*K + k]     (B is stored N x K row-major, i.e. K x N
 *                                   column-major, the layout the fp16
 *                                   512^3 workload states)
 * s      = 1 for fp16/bf16, 1/(scale_a*scale_b) for e4m3 (per-tensor scaling).
 *
 * The element values are the exact reals the input bits encode; fp64 holds
 * every fp16, bf16 and e4m3 value and every product of two of them exactly.
 *
 * A companion routine returns s * sum_k |a[i,k]|*|b[k,j]|, the normaliser of
 * the relative-error metric the parity tests use.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2 };

/* IEEE 754-2008 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent field 0 = zero/subnormal (value = frac * 2^-24), 31 =
 * inf/NaN. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 (1 sign, 8 exponent bits with
 * bias 127, 7 fraction bits). */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);
    return sign ? -v : v;
}

/* OCP 8-bit floating point, E4M3 ("e4m3fn"): 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities; S.1111.111 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.  Exponent field 0 = subnormal, value
 * m * 2^-9. */
double oracle_decode_e4m3(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int m = b & 0x7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

static double decode_at(const void *p, int dtype, size_t idx)
{
    if (dtype == ORACLE_E4M3)
        return oracle_decode_e4m3(((const uint8_t *)p)[idx]);
    if (dtype == ORACLE_BF16)
        return oracle_decode_bf16(((const uint16_t *)p)[idx]);
    return oracle_decode_f16(((const uint16_t *)p)[idx]);
}

/* Decode n raw elements into fp64. */
static double *decode_all(const void *p, int dtype, size_t n)
{
    double *out = (double *)malloc((n ? n : 1) * sizeof(double));
    if (!out)
        return NULL;
    for (size_t t = 0; t < n; ++t)
        out[t] = decode_at(p, dtype, t);
    return out;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int valid_args(int64_t M, int64_t N, int64_t K, int dtype)
{
    return M >= 0 && N >= 0 && K >= 0 && dtype >= ORACLE_F16 && dtype <= ORACLE_E4M3;
}

/*
 * Full product.  C and Cabs (either may be NULL) are M x N row-major fp64.
 * nthreads <= 0 uses every host thread; rows are split across threads, each
 * output keeps the serial k order.  Returns 0, or -1 on bad arguments or
 * allocation failure.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K, const void *A, const void *B, int dtype,
                double s, double *C, double *Cabs, int nthreads)
{
    if (!valid_args(M, N, K, dtype))
        return -1;
    double *a = decode_all(A, dtype, (size_t)M * (size_t)K);
    double *b = decode_all(B, dtype, (size_t)N * (size_t)K);
    if (!a || !b) {
        free(a);
        free(b);
        return -1;
    }
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < M; ++i) {
        const double *ai = a + (size_t)i * (size_t)K;
        for (int64_t j = 0; j < N; ++j) {
            const double *bj = b + (size_t)j * (size_t)K;
            double acc = 0.0, acc_abs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                acc += ai[k] * bj[k];
                acc_abs += fabs(ai[k]) * fabs(bj[k]);
            }
            if (C)
                C[(size_t)i * (size_t)N + (size_t)j] = s * acc;
            if (Cabs)
                Cabs[(size_t)i * (size_t)N + (size_t)j] = fabs(s) * acc_abs;
        }
    }
    free(a);
    free(b);
    return 0;
}

/*
 * The same definition evaluated only at the n positions (ii[t], jj[t]); used
 * where the full product is too slow for the CPU.  Elements are decoded on the
 * fly from the raw buffers.  Returns 0, or -1 on bad arguments (an index out of
 * range included).
 */
int oracle_gemm_sampled(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                        int dtype, double s, int64_t n, const int64_t *ii, const int64_t *jj,
                        double *C, double *Cabs, int nthreads)
{
    if (!valid_args(M, N, K, dtype) || n < 0)
        return -1;
    for (int64_t t = 0; t < n; ++t)
        if (ii[t] < 0 || ii[t] >= M || jj[t] < 0 || jj[t] >= N)
            return -1;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
#else
    (void)nthreads;
#endif
    for (int64_t t = 0; t < n; ++t) {
        size_t rowa = (size_t)ii[t] * (size_t)K;
        size_t rowb = (size_t)jj[t] * (size_t)K;
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double x = decode_at(A, dtype, rowa + (size_t)k);
            double y = decode_at(B, dtype, rowb + (size_t)k);
            acc += x * y;
            acc_abs += fabs(x) * fabs(y);
        }
        if (C)
            C[t] = s * acc;
        if (Cabs)
            Cabs[t] = fabs(s) * acc_abs;
    }
    return 0;
}
