"""CPU oracle for the persistent tile-scheduled GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA path and never imports it.

Modules:
  gemm   -- C[i,j] = s * sum_k a[i,k]*b[k,j] in fp64: a C triple loop
            (``oracle.c``), a numpy version and a pure-Python loop, plus the
            relative-error metric the parity tests use.
  sched  -- what the three tile schedulers compute: the GROUP_SIZE_M
            swizzle, the static and non-persistent tile assignments, and a
            replay model of Cluster Launch Control work stealing.
"""
