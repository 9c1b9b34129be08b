"""The C ABI on a machine without a GPU: the library builds, loads, exports
every function include/pts_gemm.h declares, its structs match the Python
binding byte for byte, and calls that need no device fail cleanly."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import persistent_tile_scheduled_gb300 as pts
from persistent_tile_scheduled_gb300 import gemm as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pts_gemm.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert _declared_functions() == sorted(g.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = pts.load()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pts._build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (gemm_\w+)", out))
    assert set(_declared_functions()) <= exported


def test_status_strings():
    for s in range(6):
        assert pts.gemm_status_string(s)
    assert pts.gemm_status_string(99) == "unknown status"


def test_calls_without_a_handle_are_rejected():
    lib = pts.load()
    assert lib.gemm_run(None, 8, 8, 8, None, None, None, 0, 0, 1.0, 1.0, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_create(None, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_destroy(None) == g.GEMM_OK
    info = g.gemm_launch_info_t()
    assert lib.gemm_query(None, 8, 8, 8, 0, 0, ctypes.byref(info)) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_run_grouped(None, None, 0, 0, 0, None) == g.GEMM_ERR_INVALID_ARG
    assert lib.gemm_query_grouped(None, None, 0, 0, 0, ctypes.byref(info)) == g.GEMM_ERR_INVALID_ARG


def test_bad_options_are_rejected_before_touching_a_device():
    lib = pts.load()
    h = ctypes.c_void_p()
    for bad in (g.make_opts(cta_group=3), g.make_opts(stages=1), g.make_opts(stages=99),
                g.make_opts(group_size_m=-1), g.make_opts(debug_flags=0x80), g.make_opts(prefetch=-2),
                g.make_opts(prefetch=65), g.make_opts(split=3), g.make_opts(split_k=2), g.make_opts(split_k=-2),
                g.make_opts(split=2, split_k=1), g.make_opts(overlap_launch=1), g.make_opts(overlap_launch=-2),
                g.make_opts(epilogue=3), g.make_opts(max_clusters=-1), g.make_opts(group_order=3),
                g.make_opts(group_order=-1), g.make_opts(tile_n=64), g.make_opts(tile_n=512),
                g.make_opts(tile_n=128, split=4),
                g.make_opts(tile_n=128, split_k=1), g.make_opts(clc_depth=3), g.make_opts(clc_depth=-1)):
        assert lib.gemm_create(ctypes.byref(h), 0, ctypes.byref(bad)) == g.GEMM_ERR_INVALID_ARG
        assert h.value is None


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="a GPU is present")
def test_create_without_a_gpu_fails_cleanly():
    h = ctypes.c_void_p()
    st = pts.load().gemm_create(ctypes.byref(h), 0, None)
    assert st in (g.GEMM_ERR_CUDA, g.GEMM_ERR_UNSUPPORTED) and h.value is None


def test_struct_layouts_match_the_header():
    src = r"""
    #include <stdio.h>
    #include <stddef.h>
    #include "pts_gemm.h"
    int main(void) {
      printf("%zu %zu %zu %zu\n", sizeof(gemm_opts_t), offsetof(gemm_opts_t, debug_flags),
             offsetof(gemm_opts_t, fault_arg), offsetof(gemm_opts_t, timeout_ns));
      printf("%zu %zu %zu\n", sizeof(gemm_tile_record_t), offsetof(gemm_tile_record_t, smid),
             offsetof(gemm_tile_record_t, group));
      printf("%zu %zu %zu %zu\n", sizeof(gemm_group_problem_t), offsetof(gemm_group_problem_t, A),
             offsetof(gemm_group_problem_t, scale_a), (size_t)GEMM_GROUPED_MAX_PROBLEMS);
      printf("%zu %zu %zu %zu\n", sizeof(gemm_launch_info_t), offsetof(gemm_launch_info_t, tiles_m),
             offsetof(gemm_launch_info_t, grid_ctas), offsetof(gemm_launch_info_t, threads));
      printf("%zu %zu %zu %zu\n", offsetof(gemm_launch_info_t, sk_tiles), offsetof(gemm_launch_info_t, work_items),
             offsetof(gemm_launch_info_t, units), offsetof(gemm_launch_info_t, ctas_per_sm));
      printf("%zu %zu %zu\n", offsetof(gemm_opts_t, tile_n), offsetof(gemm_opts_t, clc_depth),
             offsetof(gemm_launch_info_t, tail_tiles));
      return 0;
    }
    """
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    got = [int(v) for v in out]
    want = [ctypes.sizeof(g.gemm_opts_t), g.gemm_opts_t.debug_flags.offset, g.gemm_opts_t.fault_arg.offset,
            g.gemm_opts_t.timeout_ns.offset,
            ctypes.sizeof(g.gemm_tile_record_t), g.gemm_tile_record_t.smid.offset, g.gemm_tile_record_t.group.offset,
            ctypes.sizeof(g.gemm_group_problem_t), g.gemm_group_problem_t.A.offset,
            g.gemm_group_problem_t.scale_a.offset, g.GEMM_GROUPED_MAX_PROBLEMS,
            ctypes.sizeof(g.gemm_launch_info_t), g.gemm_launch_info_t.tiles_m.offset,
            g.gemm_launch_info_t.grid_ctas.offset, g.gemm_launch_info_t.threads.offset,
            g.gemm_launch_info_t.sk_tiles.offset, g.gemm_launch_info_t.work_items.offset,
            g.gemm_launch_info_t.units.offset, g.gemm_launch_info_t.ctas_per_sm.offset,
            g.gemm_opts_t.tile_n.offset, g.gemm_opts_t.clc_depth.offset, g.gemm_launch_info_t.tail_tiles.offset]
    assert got == want


def test_no_cpu_fallback_in_the_package():
    """The product package never imports the oracle or multiplies matrices on the host."""
    pkg = os.path.join(ROOT, "persistent_tile_scheduled_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                text = open(os.path.join(dirpath, f)).read()
                for banned in ("oracle", "matmul", " @ ", "torch.mm", "einsum"):
                    assert banned not in text, (f, banned)


def test_group_problem_marshalling():
    """The binding packs (M, N, K, A, B, C[, scale_a, scale_b]) into the C
    struct field by field; raw addresses pass through unchanged."""
    arr = g.group_array([(3, 8, 16, 0x1000, 0x2000, 0x3000), (0, 64, 0, 0, 0, 0x4000, 2.0, 0.5)])
    assert arr.count == 2
    a, b = arr.arr[0], arr.arr[1]
    assert (a.M, a.N, a.K, a.A, a.B, a.C, a.scale_a, a.scale_b) == (3, 8, 16, 0x1000, 0x2000, 0x3000, 1.0, 1.0)
    assert (b.M, b.N, b.K, b.A, b.B, b.C, b.scale_a, b.scale_b) == (0, 64, 0, None, None, 0x4000, 2.0, 0.5)
    assert g.group_array(arr) is arr
    assert g.group_array([]).count == 0
