"""Persistent, tile-scheduled GEMM for GB300 (sm_103a): Python binding.

The compute path is libpts_gemm.so (hand-written CUDA, see csrc/); this
package only builds it and marshals arguments into its C ABI
(include/pts_gemm.h).  Importing the package does not load the library; the
first call does, and raises if it cannot.
"""
from .gemm import (GEMM_BF16, GEMM_DEBUG_CLC_STOP_AT, GEMM_DEBUG_FAULT_SKIP_TMA, GEMM_DEBUG_RECORDS, GEMM_E4M3, GEMM_F16,  # noqa: F401
                   GEMM_SCHED_CLC, GEMM_SCHED_NONPERSISTENT, GEMM_SCHED_STATIC, SCHEDS, GemmError,
                   gemm_check, gemm_create, gemm_destroy, gemm_query, gemm_query_grouped, gemm_read_debug, gemm_run,
                   gemm_run_grouped, gemm_run_host, gemm_run_host_batch, gemm_run_noalloc, gemm_status_string, gemm_tensor_peak_probe, load,
                   make_opts)
from ._build import build  # noqa: F401
