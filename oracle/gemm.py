"""fp64 oracle for C = A . B over fp16 / bf16 / e4m3 inputs (test infrastructure).

Only tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs use
this module.  It never imports the CUDA package.

Definition followed (the GEMM that "question about persistent kernel concept"
splits into output tiles, and that "[Persistent] Performance on
09-persistent-matmul on A100 worse than non-persistent" benchmarks in fp16):

    C[i, j] = s * sum_{k < K} a[i, k] * b[k, j]

with ``a[i, k] = A[i*K + k]`` (A: M x K row-major), ``b[k, j] = B[j*K + k]``
(B stored N x K, i.e. K x N column-major) and ``s = 1`` for fp16 / bf16,
``s = 1 / (scale_a * scale_b)`` for e4m3 inputs that were scaled per tensor
before rounding.  The element values are the exact reals the stored bits
encode; every product of two such values is exact in fp64.

Three independent evaluations of the same definition:
  * ``gemm`` / ``gemm_sampled`` -- the C triple loop in ``oracle.c``
  * ``gemm_numpy`` -- decode with numpy bit arithmetic, then one fp64 matmul
  * ``gemm_loops`` -- a pure-Python triple loop, for tiny shapes only
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F16, BF16, E4M3 = 0, 1, 2
DTYPES = {"f16": F16, "fp16": F16, "bf16": BF16, "e4m3": E4M3, "fp8": E4M3}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (OpenMP when gcc has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, dp, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
        lib.oracle_gemm.argtypes = [i64, i64, i64, vp, vp, ctypes.c_int, ctypes.c_double,
                                    vp, vp, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_sampled.argtypes = [i64, i64, i64, vp, vp, ctypes.c_int, ctypes.c_double,
                                            i64, vp, vp, vp, vp, ctypes.c_int]
        lib.oracle_gemm_sampled.restype = ctypes.c_int
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_f16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_max_threads.restype = ctypes.c_int
        _ = dp
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _bits(x: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint8 if dtype == E4M3 else np.uint16
    x = np.ascontiguousarray(x)
    if x.dtype != want:
        raise TypeError(f"expected raw {want.__name__} bits, got {x.dtype}")
    return x


def decode_c(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode raw bits with the C decoders (one call per element; small arrays)."""
    lib = _load()
    fn = {F16: lib.oracle_decode_f16, BF16: lib.oracle_decode_bf16, E4M3: lib.oracle_decode_e4m3}[dtype]
    flat = np.asarray(bits).ravel()
    return np.array([fn(int(v)) for v in flat], dtype=np.float64).reshape(np.shape(bits))


def gemm(M, N, K, A_bits, B_bits, dtype, s=1.0, nthreads=0, with_abs=True):
    """Full product via the C triple loop.  Returns (C, Cabs) as M x N fp64."""
    A_bits, B_bits = _bits(A_bits, dtype), _bits(B_bits, dtype)
    assert A_bits.size == M * K and B_bits.size == N * K
    C = np.empty((M, N), np.float64)
    Cabs = np.empty((M, N), np.float64) if with_abs else None
    rc = _load().oracle_gemm(M, N, K, A_bits.ctypes.data, B_bits.ctypes.data, dtype, float(s),
                             C.ctypes.data, Cabs.ctypes.data if with_abs else None, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return C, Cabs


def gemm_sampled(M, N, K, A_bits, B_bits, dtype, ii, jj, s=1.0, nthreads=0):
    """The definition at positions (ii[t], jj[t]) only.  Returns (C, Cabs) of length n."""
    A_bits, B_bits = _bits(A_bits, dtype), _bits(B_bits, dtype)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    n = ii.size
    C = np.empty(n, np.float64)
    Cabs = np.empty(n, np.float64)
    rc = _load().oracle_gemm_sampled(M, N, K, A_bits.ctypes.data, B_bits.ctypes.data, dtype,
                                     float(s), n, ii.ctypes.data, jj.ctypes.data, C.ctypes.data,
                                     Cabs.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_sampled rejected its arguments")
    return C, Cabs


# ---------------------------------------------------------------------------
# numpy decoders: the same format definitions written with array bit fields.
# ---------------------------------------------------------------------------

def decode_np(bits: np.ndarray, dtype: int) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64)
    if dtype == F16:
        sign, e, f = (b >> 15) & 1, (b >> 10) & 0x1F, b & 0x3FF
        v = np.where(e == 0, np.ldexp(f.astype(np.float64), -24),
                     np.ldexp((1024 + f).astype(np.float64), (e - 25).astype(np.int32)))
        v = np.where(e == 31, np.where(f == 0, np.inf, np.nan), v)
    elif dtype == BF16:
        sign, e, f = (b >> 15) & 1, (b >> 7) & 0xFF, b & 0x7F
        v = np.where(e == 0, np.ldexp(f.astype(np.float64), -133),
                     np.ldexp((128 + f).astype(np.float64), (e - 134).astype(np.int32)))
        v = np.where(e == 255, np.where(f == 0, np.inf, np.nan), v)
    elif dtype == E4M3:
        sign, e, m = (b >> 7) & 1, (b >> 3) & 0xF, b & 0x7
        v = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                     np.ldexp((8 + m).astype(np.float64), (e - 10).astype(np.int32)))
        v = np.where((e == 15) & (m == 7), np.nan, v)
    else:
        raise ValueError(dtype)
    return np.where(sign == 1, -v, v)


def gemm_numpy(M, N, K, A_bits, B_bits, dtype, s=1.0):
    """Decode, then one fp64 matmul (a library primitive as the only step)."""
    a = decode_np(np.asarray(A_bits).reshape(M, K), dtype)
    b = decode_np(np.asarray(B_bits).reshape(N, K), dtype)   # b[j, k]
    C = s * (a @ b.T)
    Cabs = abs(s) * (np.abs(a) @ np.abs(b).T)
    return C, Cabs


# ---------------------------------------------------------------------------
# pure-Python decoders + triple loop (tiny shapes): a third, separate route.
# ---------------------------------------------------------------------------

def _py_decode(v: int, dtype: int) -> float:
    if dtype == F16:
        sign, e, f, bias, mbits, emax = v >> 15, (v >> 10) & 31, v & 1023, 15, 10, 31
    elif dtype == BF16:
        sign, e, f, bias, mbits, emax = v >> 15, (v >> 7) & 255, v & 127, 127, 7, 255
    else:
        sign, e, f, bias, mbits, emax = v >> 7, (v >> 3) & 15, v & 7, 7, 3, None
        if e == 15 and f == 7:
            return float("nan")
    if emax is not None and e == emax:
        x = float("inf") if f == 0 else float("nan")
    elif e == 0:
        x = f / (1 << mbits) * 2.0 ** (1 - bias)
    else:
        x = (1 + f / (1 << mbits)) * 2.0 ** (e - bias)
    return -x if sign else x


def gemm_loops(M, N, K, A_bits, B_bits, dtype, s=1.0):
    A = [int(v) for v in np.asarray(A_bits).ravel()]
    B = [int(v) for v in np.asarray(B_bits).ravel()]
    C = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += _py_decode(A[i * K + k], dtype) * _py_decode(B[j * K + k], dtype)
            C[i][j] = s * acc
    return np.array(C, dtype=np.float64).reshape(M, N)


# ---------------------------------------------------------------------------
# comparison metric
# ---------------------------------------------------------------------------

OUT_UNIT_ROUNDOFF = {F16: 2.0 ** -11, BF16: 2.0 ** -8}   # RNE to the output format: |err| <= u |x|


def rel_err(C_test, C_ref, C_abs, out_u: float = 0.0):
    """max (|C_test - C_ref| - out_u * |C_ref|)+ / (s * sum_k |a||b|).

    ``out_u`` is the unit roundoff of the output format (2^-11 for fp16,
    2^-8 for bf16): rounding the exact result to that format may move it by up
    to out_u * |C_ref|, which no kernel can avoid, so that much is not charged.
    ``out_u = 0`` gives the plain normalised error.  Elements whose normaliser
    is 0 must be exactly 0 in C_test; any that are not make the error infinite.
    """
    C_test = np.asarray(C_test, np.float64)
    C_ref = np.asarray(C_ref, np.float64)
    C_abs = np.asarray(C_abs, np.float64)
    zero = C_abs == 0
    if np.any(zero & (C_test != 0)):
        return float("inf")
    if not np.all(np.isfinite(C_test[~zero])):
        return float("inf")
    if not np.any(~zero):
        return 0.0
    d = np.abs(C_test[~zero] - C_ref[~zero]) - out_u * np.abs(C_ref[~zero])
    return float(max(np.max(d / C_abs[~zero]), 0.0))
