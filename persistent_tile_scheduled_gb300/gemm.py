"""Python binding of the C ABI in include/pts_gemm.h (argument marshalling only).

Every function keeps the C name and order of arguments; tensors may be passed
where the C call takes a pointer (their ``data_ptr()`` is used).  All compute
happens in libpts_gemm.so; if the library cannot be loaded the call raises --
there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

GEMM_F16, GEMM_BF16, GEMM_E4M3 = 0, 1, 2
GEMM_SCHED_NONPERSISTENT, GEMM_SCHED_STATIC, GEMM_SCHED_CLC = 0, 1, 2
SCHEDS = {"nonpersistent": 0, "static": 1, "clc": 2}
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT, GEMM_ERR_COVERAGE = range(6)
GEMM_DEBUG_RECORDS = 0x1
GEMM_DEBUG_CLC_STOP_AT = 0x2
GEMM_DEBUG_FAULT_SKIP_TMA = 0x4

EXPORTED = ("gemm_create", "gemm_run", "gemm_run_host", "gemm_query", "gemm_check",
            "gemm_read_debug", "gemm_destroy", "gemm_status_string", "gemm_run_noalloc",
            "gemm_run_host_batch", "gemm_run_grouped", "gemm_query_grouped", "gemm_tensor_peak_probe")
GEMM_NOALLOC_MAX_WORK_ITEMS = 16384
GEMM_GROUPED_MAX_PROBLEMS = 65536


class gemm_opts_t(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int), ("group_size_m", ctypes.c_int), ("stages", ctypes.c_int),
                ("max_clusters", ctypes.c_int), ("debug_flags", ctypes.c_uint), ("fault_arg", ctypes.c_int),
                ("timeout_ns", ctypes.c_ulonglong), ("split", ctypes.c_int), ("split_k", ctypes.c_int),
                ("prefetch", ctypes.c_int), ("overlap_launch", ctypes.c_int), ("epilogue", ctypes.c_int),
                ("group_order", ctypes.c_int), ("tile_n", ctypes.c_int), ("clc_depth", ctypes.c_int)]


class gemm_tile_record_t(ctypes.Structure):
    _fields_ = [("visits", ctypes.c_uint32), ("tile", ctypes.c_uint32), ("n_off", ctypes.c_uint32),
                ("n_len", ctypes.c_uint32), ("owner", ctypes.c_uint32), ("iter", ctypes.c_uint32),
                ("smid", ctypes.c_uint32), ("t_mma_start", ctypes.c_uint32), ("t_acc_full", ctypes.c_uint32),
                ("t_stored", ctypes.c_uint32), ("kb_begin", ctypes.c_uint32), ("kb_end", ctypes.c_uint32),
                ("group", ctypes.c_uint32)]


class gemm_launch_info_t(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("cta_group", ctypes.c_int), ("stages", ctypes.c_int), ("tiles_m", ctypes.c_int64),
                ("tiles_n", ctypes.c_int64), ("tiles", ctypes.c_int64), ("grid_ctas", ctypes.c_int64),
                ("max_active_clusters", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("threads", ctypes.c_int),
                ("split", ctypes.c_int), ("split_k", ctypes.c_int), ("sk_tiles", ctypes.c_int64),
                ("sk_units", ctypes.c_int64), ("work_items", ctypes.c_int64), ("units", ctypes.c_int64),
                ("ctas_per_sm", ctypes.c_int), ("tail_tiles", ctypes.c_int64)]


class gemm_host_problem_t(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("A", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("dtype", ctypes.c_int), ("scale_a", ctypes.c_float),
                ("scale_b", ctypes.c_float)]


class gemm_group_problem_t(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("A", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("scale_a", ctypes.c_float),
                ("scale_b", ctypes.c_float)]


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {gemm_status_string(status)} (status {status})")


_lib = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libpts_gemm.so (building it first if allowed); raise if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not _build.up_to_date():
        if not build_if_missing and not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        if build_if_missing:
            _build.build()
    lib = ctypes.CDLL(path)
    vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    st = ctypes.c_int
    lib.gemm_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.POINTER(gemm_opts_t)]
    lib.gemm_create.restype = st
    lib.gemm_run.argtypes = [vp, i64, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int, f32, f32, vp]
    lib.gemm_run.restype = st
    lib.gemm_run_host.argtypes = [vp, i64, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int, f32, f32, vp]
    lib.gemm_run_host.restype = st
    lib.gemm_run_host_batch.argtypes = [vp, ctypes.POINTER(gemm_host_problem_t), i64, ctypes.c_int, vp]
    lib.gemm_run_host_batch.restype = st
    lib.gemm_query.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(gemm_launch_info_t)]
    lib.gemm_query.restype = st
    lib.gemm_run_grouped.argtypes = [vp, ctypes.POINTER(gemm_group_problem_t), i64, ctypes.c_int, ctypes.c_int, vp]
    lib.gemm_run_grouped.restype = st
    lib.gemm_query_grouped.argtypes = [vp, ctypes.POINTER(gemm_group_problem_t), i64, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(gemm_launch_info_t)]
    lib.gemm_query_grouped.restype = st
    lib.gemm_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.gemm_check.restype = st
    lib.gemm_read_debug.argtypes = [vp, vp, ctypes.POINTER(gemm_tile_record_t), i64, ctypes.POINTER(ctypes.c_int)]
    lib.gemm_read_debug.restype = st
    lib.gemm_destroy.argtypes = [vp]
    lib.gemm_destroy.restype = st
    lib.gemm_run_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, ctypes.c_int, ctypes.c_int, f32, f32,
                                     ctypes.c_int, vp, ctypes.POINTER(ctypes.c_int)]
    lib.gemm_run_noalloc.restype = st
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gemm_tensor_peak_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, dp, dp, dp]
    lib.gemm_tensor_peak_probe.restype = st
    lib.gemm_status_string.argtypes = [ctypes.c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status: int, what: str) -> int:
    if status != GEMM_OK:
        raise GemmError(status, what)
    return status


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def make_opts(cta_group=0, group_size_m=8, stages=0, max_clusters=0, debug_flags=0, fault_arg=0,
              timeout_ns=0, split=0, split_k=0, prefetch=0, overlap_launch=0, epilogue=0,
              group_order=0, tile_n=0, clc_depth=0) -> gemm_opts_t:
    return gemm_opts_t(cta_group, group_size_m, stages, max_clusters, debug_flags, fault_arg, timeout_ns, split,
                       split_k, prefetch, overlap_launch, epilogue, group_order, tile_n, clc_depth)


def gemm_create(device: int = 0, opts: Optional[gemm_opts_t] = None) -> int:
    h = ctypes.c_void_p()
    _check(load().gemm_create(ctypes.byref(h), int(device), ctypes.byref(opts) if opts is not None else None),
           "gemm_create")
    return h.value


def gemm_run(h, M, N, K, A, B, C, dtype, sched, scale_a=1.0, scale_b=1.0, stream=None) -> int:
    return _check(load().gemm_run(h, M, N, K, _ptr(A), _ptr(B), _ptr(C), int(dtype), int(sched),
                                  float(scale_a), float(scale_b), _stream(stream)), "gemm_run")


def gemm_run_host(h, M, N, K, A, B, C, dtype, sched, scale_a=1.0, scale_b=1.0, stream=None) -> int:
    return _check(load().gemm_run_host(h, M, N, K, _ptr(A), _ptr(B), _ptr(C), int(dtype), int(sched),
                                       float(scale_a), float(scale_b), _stream(stream)), "gemm_run_host")


def gemm_run_host_batch(h, problems, sched, stream=None) -> int:
    """problems: sequence of (M, N, K, A, B, C, dtype[, scale_a, scale_b]) with
    host tensors (pinned for overlap) or raw addresses."""
    arr = (gemm_host_problem_t * max(len(problems), 1))()
    for i, q in enumerate(problems):
        M, N, K, A, B, C, dt = q[:7]
        sa, sb = (q[7], q[8]) if len(q) > 7 else (1.0, 1.0)
        arr[i] = gemm_host_problem_t(M, N, K, _ptr(A), _ptr(B), _ptr(C), int(dt), float(sa), float(sb))
    return _check(load().gemm_run_host_batch(h, arr, len(problems), int(sched), _stream(stream)),
                  "gemm_run_host_batch")


class GroupArray:
    """A problem list marshalled once into the C array gemm_run_grouped reads
    (building it costs host time per problem; a loop over the same list can
    reuse it)."""

    def __init__(self, problems):
        self.count = len(problems)
        self.arr = (gemm_group_problem_t * max(self.count, 1))()
        for i, q in enumerate(problems):
            M, N, K, A, B, C = q[:6]
            sa, sb = (q[6], q[7]) if len(q) > 6 else (1.0, 1.0)
            self.arr[i] = gemm_group_problem_t(M, N, K, _ptr(A), _ptr(B), _ptr(C), float(sa), float(sb))


def group_array(problems) -> GroupArray:
    """problems: sequence of (M, N, K, A, B, C[, scale_a, scale_b]) with
    device tensors or raw device addresses."""
    return problems if isinstance(problems, GroupArray) else GroupArray(problems)


def gemm_run_grouped(h, problems, dtype, sched, stream=None) -> int:
    """problems: a GroupArray or a sequence as group_array() takes; one launch
    for all of them."""
    g = group_array(problems)
    return _check(load().gemm_run_grouped(h, g.arr, g.count, int(dtype), int(sched), _stream(stream)),
                  "gemm_run_grouped")


def gemm_query_grouped(h, problems, dtype, sched) -> gemm_launch_info_t:
    g = group_array(problems)
    info = gemm_launch_info_t()
    _check(load().gemm_query_grouped(h, g.arr, g.count, int(dtype), int(sched), ctypes.byref(info)),
           "gemm_query_grouped")
    return info


def gemm_query(h, M, N, K, dtype, sched) -> gemm_launch_info_t:
    info = gemm_launch_info_t()
    _check(load().gemm_query(h, M, N, K, int(dtype), int(sched), ctypes.byref(info)), "gemm_query")
    return info


def gemm_check(h, stream=None):
    """Returns (status, raw device status word); never raises."""
    dev = ctypes.c_int(0)
    st = load().gemm_check(h, _stream(stream), ctypes.byref(dev))
    return st, dev.value


def gemm_read_debug(h, n_work: int, stream=None):
    """Returns (status, records, raw device status word); never raises."""
    recs = (gemm_tile_record_t * max(int(n_work), 1))()
    dev = ctypes.c_int(0)
    st = load().gemm_read_debug(h, _stream(stream), recs, int(n_work), ctypes.byref(dev))
    return st, recs, dev.value


def gemm_run_noalloc(M, N, K, A, B, C, dtype, sched, scale_a=1.0, scale_b=1.0, cta_group=1, stream=None,
                     check=False):
    """The allocation-free entry point.  Returns (status, device status word);
    never raises.  check=True makes the call synchronise and report device
    errors and coverage (the C call's device_status argument)."""
    dev = ctypes.c_int(0)
    st = load().gemm_run_noalloc(M, N, K, _ptr(A), _ptr(B), _ptr(C), int(dtype), int(sched), float(scale_a),
                                 float(scale_b), int(cta_group), _stream(stream),
                                 ctypes.byref(dev) if check else None)
    return st, dev.value


def gemm_tensor_peak_probe(device, dtype, cta_group, mmas=20000) -> dict:
    """The tensor-pipe peak probe: {"flop_per_clk_per_sm", "tflops", "sm_ghz"}."""
    f, t, g = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    _check(load().gemm_tensor_peak_probe(int(device), int(dtype), int(cta_group), int(mmas), ctypes.byref(f),
                                         ctypes.byref(t), ctypes.byref(g)), "gemm_tensor_peak_probe")
    return {"flop_per_clk_per_sm": f.value, "tflops": t.value, "sm_ghz": g.value}


def gemm_destroy(h) -> int:
    return _check(load().gemm_destroy(h), "gemm_destroy")
