"""Benchmark: GEMM TFLOP/s and fraction of tensor peak vs K, per scheduler.

Workload (the fp16 K sweep of "[Persistent] Performance on 09-persistent-matmul
on A100 worse than non-persistent": M = N = 4096, K = 128..4096 step 128,
128x256x64 tiles, GROUP_SIZE_M 8).  One step = the 32 GEMMs of the sweep, each
on its own A, B, C buffers (2.1 GB together, far above the 129 MB L2, so no
GEMM finds its operands in L2 from the step before).  The step runs once per
scheduler (non-persistent, static, CLC); the headline value is the static
persistent scheduler.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  Under torchrun every rank runs the same sweep on its own
GPU (independent replicas, no collective on the data path); times are the max
over ranks and value = all ranks' FLOPs / that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "GEMM TFLOPS & % of tensor peak vs K, per scheduler (nonpersist/static/CLC)"
UNIT = "TFLOP/s"
WORKLOAD = ("fp16 GEMM M=N=4096, K=128..4096 step 128 (32 GEMMs per step), A,B ~ N(0,1)/sqrt(K), "
            "fp32 accumulate, fp16 C, row-major A, column-major B")
SCHED_NAMES = ["nonpersistent", "static", "clc"]
TILE_DESC = {0: "128x256x64 per CTA; the library's CTA group per GEMM: single CTAs (tcgen05 cta_group::1) "
                "below 14 k-blocks per tile (K <= 832), CTA pairs (one 256x256 cta_group::2 MMA sharing B) "
                "from there",
             1: "128x256x64 per CTA (tcgen05 cta_group::1)",
             2: "128x256x64 per CTA; CTA pairs run one 256x256 tcgen05 cta_group::2 MMA and share B"}
HEADLINE = "static"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
LONG_RUN_S = 0.2    # timed regions at least this long are compared with the sustained tensor peak
KERNEL_SOURCES = ["persistent_tile_scheduled_gb300/csrc/gemm_kernel.cuh",
                  "persistent_tile_scheduled_gb300/csrc/ptx.cuh",
                  "persistent_tile_scheduled_gb300/csrc/gemm_params.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------- setup

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, rank, world, local


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, *keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "tflops", "gbs"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


def kernel_hash() -> str:
    """sha256[:16] of the kernel sources without their // comments and blank
    lines, so that a comment-only edit does not retire a profile."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profile_traffic():
    """Per-launch DRAM traffic of the GEMM kernel from the committed ncu summary,
    only if it was taken on the kernel sources as they are now."""
    path = os.path.join(ROOT, "profiles", "gemm_kernel_fp16_4096_ksweep.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_sources_sha256_16") != kernel_hash():
        return None, "stale"
    return d.get("dram_bytes_per_launch_k4096"), d.get("launch")


def profile_value(name, key):
    """A per-launch figure from a committed ncu summary (profiles/<name>),
    only if that capture was taken on the kernel sources as they are now."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_sources_sha256_16") != kernel_hash():
        return None
    return d.get(key)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float, t_end: float):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for name, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def sweep_pass(pts, h, bufs, problems, sched, stream):
    """One step: the sweep's GEMMs, one gemm_run launch each, in K order, on
    `stream` (also what a captured step holds)."""
    for p, (A, B, C) in zip(problems, bufs):
        pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, 1.0, 1.0, stream)


def time_sweep(pts, h, bufs, problems, sched, steps, warmup, stream, dist, use_graph=False):
    """Warm-up, then `steps` timed passes over the sweep (events only at step
    boundaries, so consecutive GEMMs may overlap their launches), then three
    extra passes with an event between GEMMs for the per-K breakdown.  With
    use_graph the launches of a pass are captured once in a CUDA graph and
    each step replays it (the same kernels, without the host launch cost)."""
    def one_pass():
        sweep_pass(pts, h, bufs, problems, sched, stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one_pass()
    torch.cuda.synchronize()
    st, dev = pts.gemm_check(h, stream)
    if st != 0:
        raise RuntimeError(f"device status {dev:#x} after warm-up")
    step_fn = one_pass
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one_pass()
        step_fn = graph.replay
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                step_fn()
        torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for s in range(steps):
            step_fn()
            ev[s + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(dist)
    st, dev = pts.gemm_check(h, stream)
    if st != 0:
        raise RuntimeError(f"device status {dev:#x} in the timed region")
    total_ms = ev[0].elapsed_time(ev[steps])
    # per-K breakdown (outside the timed region): every GEMM timed alone, with
    # an event on each side, right behind an untimed launch of the same shape
    # on other buffers.  So its kernel is the one that just ran -- the first
    # launch of a kernel after another one can pay up to about 3 us more (in
    # the sweep's order about 2 us on the first CTA-pair K) -- while its own
    # operands are not in L2 (a launch right behind one on the same buffers
    # would find them there: 2.5 us less at K = 128).  The untimed launch uses the next
    # problem's buffers (larger K, so large enough) or, for the last, a spare
    # set.  Seven passes, the median per K (a launch of 15-20 us timed alone
    # varies by 10 % from pass to pass).
    n = len(problems)
    pl = problems[-1]
    spare = (torch.empty_like(bufs[-1][0]), torch.empty_like(bufs[-1][1]), torch.empty_like(bufs[-1][2]))
    spare[0].copy_(bufs[-1][0])
    spare[1].copy_(bufs[-1][1])
    passes = []
    for _ in range(7):
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i, (p, (A, B, C)) in enumerate(zip(problems, bufs)):
                Aw, Bw, Cw = bufs[i + 1] if i + 1 < n else spare
                pts.gemm_run(h, p.M, p.N, p.K, Aw, Bw, Cw, p.dtype, sched, 1.0, 1.0, stream)
                kev[i][0].record(stream)
                pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, 1.0, 1.0, stream)
                kev[i][1].record(stream)
        torch.cuda.synchronize()
        passes.append([a.elapsed_time(b) for a, b in kev])
    del spare
    per_k = [statistics.median(v) for v in zip(*passes)]
    assert all(q.M == pl.M and q.N == pl.N and q.K <= pl.K for q in problems)
    return total_ms, per_k, (t0, t1)


def cpu_model() -> str:
    """The host CPU's model name (/proc/cpuinfo, else lscpu, else the machine type)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name") and ":" in line:
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name") and ":" in line:
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def cpu_baseline_sample(problems, xs, budget_s=10.0):
    """The oracle as it stands on the host cores: on all threads, whole GEMMs of
    the sweep, the largest K first, until `budget_s` seconds have been spent
    (a bounded sample of the step's own work); on one thread, a row sample of
    the largest-K GEMM."""
    from oracle import gemm as og
    order = sorted(range(len(problems)), key=lambda i: -problems[i].K)
    spent, flops, done = 0.0, 0.0, []
    for i in order:
        p, x = problems[i], xs[i]
        t0 = time.perf_counter()
        og.gemm(p.M, p.N, p.K, x.bits("A").reshape(-1), x.bits("B").reshape(-1), p.dtype, nthreads=0)
        spent += time.perf_counter() - t0
        flops += gemm_flops(p.M, p.N, p.K)
        done.append(p.K)
        if spent >= budget_s:
            break
    p, x = problems[order[0]], xs[order[0]]
    A, B = x.bits("A").reshape(-1), x.bits("B").reshape(-1)
    rows, spent1 = 1, 0.0
    while True:   # one thread: rows 0..rows-1, growing until it takes a second or 16 rows
        t0 = time.perf_counter()
        og.gemm(rows, p.N, p.K, A[: rows * p.K], B, p.dtype, nthreads=1)
        spent1 = time.perf_counter() - t0
        if spent1 > 1.0 or rows >= 16:
            break
        rows *= 4
    v_one = gemm_flops(rows, p.N, p.K) / spent1 / 1e12
    ks = ", ".join(str(k) for k in done)
    return {"value": flops / spent / 1e12, "unit": UNIT, "cores": og.max_threads(), "kind": "oracle",
            "sample": f"{len(done)} whole GEMMs of the sweep, the largest K first (M = N = 4096, K = {ks}; "
                      f"fp64 triple loop over all outputs and all K), {spent:.1f} s",
            "single_thread": {"value": v_one, "unit": UNIT, "cores": 1,
                              "sample": f"rows 0..{rows - 1} of the K = {p.K} GEMM, {spent1:.1f} s"},
            "cpu_model": cpu_model(), "nproc": os.cpu_count()}


def oracle_full_configs():
    """The oracle as it stands, whole GEMMs, on all host threads: the small
    configuration (fp16 512^3), the fp16 sweep's two ends (4096^2 x 128 and
    x 4096) and e4m3 8192^3 (about 1.1 TFLOP of fp64 work).  A measurement of
    the CPU baseline on full problems, not part of the default run."""
    from oracle import gemm as og
    rows = []
    for p in wl.fp16_512() + wl.fp16_4096_ksweep([128, 4096]) + wl.e4m3_8192():
        x = wl.make_inputs(p)
        t0 = time.perf_counter()
        og.gemm(p.M, p.N, p.K, x.bits("A").reshape(-1), x.bits("B").reshape(-1), p.dtype,
                1.0 / (float(x.scale_a) * float(x.scale_b)) if p.dtype == wl.E4M3 else 1.0, nthreads=0)
        dt = time.perf_counter() - t0
        rows.append({"problem": p.name, "M": p.M, "N": p.N, "K": p.K, "seconds": round(dt, 3),
                     "tflops": round(gemm_flops(p.M, p.N, p.K) / dt / 1e12, 5)})
        log(f"oracle {p.name}: {dt:.2f} s")
    return {"oracle_full": rows, "cores": og.max_threads(), "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "kind": "oracle", "note": "fp64 triple loop over every output and every k, with sum |a||b| beside it"}


def run_ours(args, dist, rank, world, local):
    import persistent_tile_scheduled_gb300 as pts
    torch.cuda.set_device(local)
    pts.load(build_if_missing=False)
    problems = wl.fp16_4096_ksweep(args.ks)
    log(f"[rank {rank}] generating {len(problems)} inputs ...")
    xs = [wl.make_inputs(p) for p in problems]
    bufs = [(x.A.cuda(), x.B.cuda(), torch.empty(x.problem.M, x.problem.N, dtype=torch.float16, device="cuda"))
            for x in xs]
    stream = torch.cuda.Stream()
    flops_step = sum(gemm_flops(p.M, p.N, p.K) for p in problems)

    per_sched = {}
    clocks = None
    h = pts.gemm_create(local, pts.make_opts(cta_group=args.cta_group, epilogue=args.epilogue, split_k=args.split_k))
    try:
        for si, name in enumerate(SCHED_NAMES):
            if name not in args.scheds:
                continue
            sampler = ClockSampler(local) if name == HEADLINE else None
            if sampler:
                sampler.__enter__()
            total_ms, per_k, (t0, t1) = time_sweep(pts, h, bufs, problems, si, args.steps, args.warmup, stream, dist,
                                                   use_graph=args.graph)
            if sampler:
                sampler.__exit__(None, None, None)
                clocks = sampler.summary(t0, t1)
            total_ms = max_over_ranks(dist, total_ms)
            ms_step = total_ms / args.steps
            per_sched[name] = {
                "value": world * flops_step / (ms_step * 1e-3) / 1e12,
                "ms_per_step": ms_step,
                "per_k_tflops_isolated": [round(gemm_flops(p.M, p.N, p.K) / (t * 1e-3) / 1e12, 1)
                                          for p, t in zip(problems, per_k)],
                "per_k_ms": per_k,
            }
            log(f"[rank {rank}] {name}: {per_sched[name]['value']:.1f} TFLOP/s, {ms_step:.3f} ms/step")

        # end-to-end through the public host-buffer API (copies inside the timed region)
        e2e = None
        if args.e2e:
            e2e = end_to_end(pts, h, xs, problems, args, dist, world, flops_step, stream)
        peaks, peaks_src = load_peaks()
        target = target_8192(pts, local, stream, peaks, peaks_src) if args.square and rank == 0 else None
        small = small_points(pts, local, stream, peaks) if args.extras and rank == 0 else None
        sweep8 = bf16_8192_sweep(pts, local, stream, peaks) if args.extras and rank == 0 else None
        extras = extra_configs(pts, local, stream) if args.extras and rank == 0 else None
    finally:
        pts.gemm_destroy(h)
    line = finish(args, per_sched, problems, world, clocks, e2e, None, rank, xs, flops_step)
    if target is not None:
        line["bf16_8192_cubed"] = target
    if small is not None:
        line["fp16_512"] = small.pop("fp16_512")
        line["fp16_4096_small_k"] = small
    if sweep8 is not None:
        line["bf16_8192_ksweep"] = sweep8
    if extras is not None:
        line["other_configs"] = extras
    if args.square and rank == 0:
        # context for the tensor peak (the roofline keeps the denominator above): the
        # library's MMA-only probe, FLOP per SM clock and the aggregate at the clock it ran at
        line["peaks"]["tensor_probe"] = {
            name: pts.gemm_tensor_peak_probe(local, dt, 2, 100000)
            for name, dt in (("bf16", wl.BF16), ("e4m3", wl.E4M3))}
    return line


def point_roofline(p, ms, peaks):
    """Roofline of one GEMM: attainable = min(dense tensor peak, I * HBM
    bandwidth) with I = 2MNK / (compulsory bytes e*(MK + NK) + 2MN); e4m3 runs
    at twice the bf16 tensor rate."""
    tensor = peak_value(peaks, "bf16_tflops", "bf16_tflops_burst")
    hbm = peak_value(peaks, "hbm_gbs", "hbm_GBs")
    fl = gemm_flops(p.M, p.N, p.K)
    e = 1.0 if p.dtype == wl.E4M3 else 2.0
    q = e * (p.M * p.K + p.N * p.K) + 2.0 * p.M * p.N
    if not tensor or not hbm:
        return {"tflops": round(fl / (ms * 1e-3) / 1e12, 1)}
    t_peak = tensor * (2.0 if p.dtype == wl.E4M3 else 1.0)
    attain = min(t_peak, fl / q * hbm * 1e-3)
    got = fl / (ms * 1e-3) / 1e12
    return {"tflops": round(got, 1), "bound": "tensor" if attain == t_peak else "hbm",
            "attainable_tflops": round(attain, 1), "frac": round(got / attain, 3)}


def time_launches(pts, h, p, A, B, C, sa, sb, sched, stream, reps, flush=None):
    """Median CUDA-event time (ms) of one gemm_run launch: back to back on the
    same buffers, or, with `flush` (a buffer larger than L2), each launch
    after the flush buffer was overwritten so that it starts with a cold L2."""
    for _ in range(3):
        pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, sa, sb, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            if flush is not None:
                flush.zero_()
            e0.record(stream)
            pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, sa, sb, stream)
            e1.record(stream)
    torch.cuda.synchronize()
    if pts.gemm_check(h, stream)[0] != 0:
        raise RuntimeError(f"device error in {p.name}")
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)


def target_8192(pts, dev, stream, peaks, peaks_src, reps=10):
    """bf16 M = N = K = 8192 (the largest point of the bf16 sweep) per
    scheduler with the library's defaults (CTA pairs at this K), each a median
    of back-to-back launches on 268 MB of A and B (above the 129 MB L2); its
    own clock record and roofline.  Single CTAs and pairs forced are listed
    too."""
    p = wl.bf16_8192_ksweep([8192])[0]
    A, B, sa, sb = device_inputs(p, 3000 + 8192)
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    out = {"workload": "bf16 GEMM M=N=K=8192, A,B ~ N(0,1)/sqrt(K), fp32 accumulate, bf16 C"}
    h = pts.gemm_create(dev, None)
    sampler = ClockSampler(dev)
    try:
        out["cta_group"] = int(pts.gemm_query(h, p.M, p.N, p.K, p.dtype, 1).cta_group)
        sampler.__enter__()
        t0 = time.time()
        for si, name in enumerate(SCHED_NAMES):
            ms = time_launches(pts, h, p, A, B, C, sa, sb, si, stream, reps)
            out[name] = round(gemm_flops(p.M, p.N, p.K) / (ms * 1e-3) / 1e12, 1)
            out[name + "_ms"] = round(ms, 4)
        t1 = time.time()
        sampler.__exit__(None, None, None)
        out["clocks"] = sampler.summary(t0, t1)
    finally:
        pts.gemm_destroy(h)
    for cg in (1, 2):
        h = pts.gemm_create(dev, pts.make_opts(cta_group=cg))
        try:
            for si, name in enumerate(SCHED_NAMES):
                ms = time_launches(pts, h, p, A, B, C, sa, sb, si, stream, 5)
                out[f"cg{cg}_{name}"] = round(gemm_flops(p.M, p.N, p.K) / (ms * 1e-3) / 1e12, 1)
        finally:
            pts.gemm_destroy(h)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tensor = peak_value(peaks, "bf16_tflops", "bf16_tflops_burst")
    mhz_max = peak_value(peaks, "sm_max_mhz") or 2070.0
    theo = sms * 8192 * mhz_max * 1e6 / 1e12      # dense FLOP per SM clock pinned by the probe test
    mhz = out["clocks"].get("sm_mhz")
    best = max(out["static"], out["clc"])
    traffic = profile_value("gemm_kernel_bf16_8192.json", "dram_bytes_per_launch")
    out["roofline"] = {
        "bound": "tensor", "achieved": out["static"], "peak": tensor, "unit": UNIT,
        "frac": round(out["static"] / tensor, 4) if tensor else None,
        "traffic": traffic, "peak_source": f"{peaks_src} bf16 dense, burst",
        "achieved_def": "2*8192^3 / median CUDA-event time of one launch, static scheduler, library defaults",
        "theoretical_tflops_at_max_clock": round(theo, 1),
        "frac_of_theoretical": round(out["static"] / theo, 4),
        "frac_of_theoretical_at_sampled_clock": (round(out["static"] / (sms * 8192 * mhz * 1e6 / 1e12), 4)
                                                 if mhz else None),
        "best_persistent_frac_of_theoretical": round(best / theo, 4),
    }
    out["persistent_ahead"] = min(out["static"], out["clc"]) > out["nonpersistent"]
    del A, B, C
    return out


def small_points(pts, dev, stream, peaks, reps=20):
    """fp16 512^3 (U[-1,1], 8 tiles) and the small-K end of the fp16 4096
    sweep, per scheduler, library defaults: back to back on the same buffers
    (the data stays in L2 between launches) and with L2 flushed before every
    launch (a 256 MB buffer overwritten; not timed)."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    h = pts.gemm_create(dev, None)
    try:
        for p in wl.fp16_512() + wl.fp16_4096_ksweep([128, 256, 384, 512]):
            x = wl.make_inputs(p)
            A, B = x.A.cuda(), x.B.cuda()
            C = torch.empty(p.M, p.N, dtype=torch.float16, device="cuda")
            torch.cuda.synchronize()
            row = {"M": p.M, "N": p.N, "K": p.K,
                   "cta_group": int(pts.gemm_query(h, p.M, p.N, p.K, p.dtype, 1).cta_group)}
            for si, name in enumerate(SCHED_NAMES):
                warm = time_launches(pts, h, p, A, B, C, 1.0, 1.0, si, stream, reps)
                cold = time_launches(pts, h, p, A, B, C, 1.0, 1.0, si, stream, reps, flush=flush)
                row[name] = {"us": round(warm * 1e3, 2), "l2_flushed_us": round(cold * 1e3, 2),
                             **point_roofline(p, warm, peaks),
                             "l2_flushed": point_roofline(p, cold, peaks)}
            out[p.name if p.name == "fp16_512" else f"K{p.K}"] = row
            del A, B, C
    finally:
        pts.gemm_destroy(h)
    del flush
    out["note"] = (f"median of {reps} launches per scheduler; 'us' back to back on the same buffers, "
                   "'l2_flushed_us' each launch after a 256 MB buffer was overwritten (L2 is 129 MB)")
    return out


def bf16_8192_sweep(pts, dev, stream, peaks, reps=5):
    """The bf16 M = N = 8192 sweep, K = 256..8192 step 256 (32 GEMMs), per
    scheduler, library defaults: TFLOP/s per K (median of back-to-back
    launches) and its fraction of the point's roofline."""
    h = pts.gemm_create(dev, None)
    out = {"K": [], "attainable_tflops": []}
    try:
        for i, p in enumerate(wl.bf16_8192_ksweep()):
            A, B, sa, sb = device_inputs(p, 6000 + i)
            C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
            out["K"].append(p.K)
            for si, name in enumerate(SCHED_NAMES):
                ms = time_launches(pts, h, p, A, B, C, sa, sb, si, stream, reps)
                r = point_roofline(p, ms, peaks)
                out.setdefault(name, []).append(r["tflops"])
                out.setdefault(name + "_frac", []).append(r.get("frac"))
            out["attainable_tflops"].append(r.get("attainable_tflops"))
            del A, B, C
    finally:
        pts.gemm_destroy(h)
    tensor = peak_value(peaks, "bf16_tflops", "bf16_tflops_burst")
    for name in SCHED_NAMES:
        out[name + "_mean"] = round(sum(out[name]) / len(out[name]), 1)
        if tensor:
            out[name + "_pct_of_tensor_peak"] = [round(100.0 * t / tensor, 1) for t in out[name]]
    out["persistent_ahead_at_every_K"] = all(
        min(s_, c_) > n_ for s_, c_, n_ in zip(out["static"], out["clc"], out["nonpersistent"]))
    out["note"] = (f"median of {reps} back-to-back launches per K; inputs drawn on the GPU from seeded "
                   "generators (parity for these shapes is in the tests)")
    return out


def end_to_end(pts, h, xs, problems, args, dist, world, flops_step, stream):
    """The step through the public host-buffer API: gemm_run_host_batch copies
    every A, B in from pinned host memory and every C back out, overlapping the
    transfers of neighbouring GEMMs with the compute; all inside the timing."""
    host = [(x.A.pin_memory(), x.B.pin_memory(),
             torch.empty(x.problem.M, x.problem.N, dtype=torch.float16).pin_memory()) for x in xs]
    batch = [(p.M, p.N, p.K, A, B, C, p.dtype) for p, (A, B, C) in zip(problems, host)]
    e2e_steps = max(1, min(args.steps, 10))
    pts.gemm_run_host_batch(h, batch, 1, stream)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        pts.gemm_run_host_batch(h, batch, 1, stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(dist, (time.perf_counter() - t0) / e2e_steps)
    bi = sum(A.numel() * A.element_size() + B.numel() * B.element_size() for A, B, _ in host)
    bo = sum(C.numel() * C.element_size() for _, _, C in host)
    return {"value": world * flops_step / e2e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "api": "gemm_run_host_batch (pinned host A, B, C; static scheduler)",
            "steps": e2e_steps, "link_gbs": round((bi + bo) / e2e_s / 1e9, 1)}


def roofline_peak(timed_s, burst, sustained):
    """The tensor peak a run of `timed_s` seconds of timed work is compared
    with: the sustained one from LONG_RUN_S on (when it is known), else the
    burst one.  Returns (peak, whether it is the sustained one)."""
    if sustained and timed_s >= LONG_RUN_S:
        return sustained, True
    return burst, False


def finish(args, per_sched, problems, world, clocks, e2e, extra, rank, xs, flops_step):
    peaks, peaks_src = load_peaks()
    tensor_peak = peak_value(peaks, "bf16_tflops", "bf16_tflops_burst")
    tensor_peak_sus = peak_value(peaks, "bf16_tflops_sustained")
    hbm = peak_value(peaks, "hbm_gbs", "hbm_GBs")
    head = per_sched.get(HEADLINE) or next(iter(per_sched.values()))
    traffic, launch = profile_traffic()
    if args.cta_group != 0 or args.epilogue != 0 or args.split_k != 0:
        traffic, launch = None, None   # the capture was taken with the library's defaults
    achieved = head["value"] / world
    # The denominator follows the length of the timed region: the burst peak for a
    # short run, the sustained one (measured over a seconds-long loop under the
    # power cap) once the timed region lasts long enough for the cap to engage
    # (on GB300: 200 steps, 0.33 s, ran at a median 2002 MHz with sw_power_cap;
    # 20 steps, 30 ms, at 2070 MHz with no throttle reason).
    timed_s = head["ms_per_step"] * args.steps / 1e3
    peak, sustained = roofline_peak(timed_s, tensor_peak, tensor_peak_sus)
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": UNIT,
                "frac": round(achieved / peak, 4) if peak else None,
                "traffic": traffic if isinstance(traffic, (int, float)) else None,
                "peak_source": (f"{peaks_src} bf16 dense (fp16 runs at the same tensor rate), "
                                f"{'sustained' if sustained else 'burst'}: the timed region lasted {timed_s:.3f} s "
                                f"({'at least' if sustained else 'under'} {LONG_RUN_S} s)"),
                "frac_burst": round(achieved / tensor_peak, 4) if tensor_peak else None,
                "frac_sustained": round(achieved / tensor_peak_sus, 4) if tensor_peak_sus else None,
                "achieved_def": "sum of 2MNK over the 32 launches of a step / the step's CUDA-event time"}
    if traffic is not None and launch:
        roofline["traffic_launch"] = launch
    per_k_roof = []
    for p, t in zip(problems, head["per_k_ms"]):
        fl = gemm_flops(p.M, p.N, p.K)
        q = 2.0 * (p.M * p.K + p.N * p.K) + 2.0 * p.M * p.N
        attain = min(tensor_peak * 1e12, fl / q * hbm * 1e9) if tensor_peak and hbm else None
        per_k_roof.append({"K": p.K, "tflops": round(fl / (t * 1e-3) / 1e12, 1),
                           "bound": "tensor" if attain == (tensor_peak or 0) * 1e12 else "hbm",
                           "attainable_tflops": round(attain / 1e12, 1) if attain else None,
                           "frac": round(fl / (t * 1e-3) / attain, 3) if attain else None})

    # the metric as named: TFLOP/s and % of the dense tensor peak vs K, per scheduler
    # (isolated launches, an event between GEMMs)
    if tensor_peak:
        for v in per_sched.values():
            v["per_k_pct_of_tensor_peak"] = [round(100.0 * t / tensor_peak, 1) for t in v["per_k_tflops_isolated"]]
            v["pct_of_tensor_peak"] = round(100.0 * v["value"] / world / tensor_peak, 2)
    line = {
        "metric": METRIC, "value": round(head["value"], 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(head["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1)/sqrt(K), rounded to fp16)",
        "config": {"workload": WORKLOAD, "tile": TILE_DESC[args.cta_group], "group_size_m": 8,
                   "cta_group": args.cta_group, "split_k": args.split_k, "sched": HEADLINE,
                   "last_wave": ("the library's choice per GEMM: with the static and CLC schedulers a partial "
                                 "last wave of at most half the clusters runs as column halves of its tiles "
                                 "below 48 k-blocks per tile (K < 3072), else the stream-K share of the last "
                                 "waves where it saves >= 20 k-blocks per cluster; the non-persistent grid "
                                 "takes only the share"
                                 if args.split_k == 0 else "as --split-k sets it"),
                   "launch": ("CUDA graph of the 32 gemm_run launches per step" if args.graph
                              else "32 gemm_run calls per step, launched one by one"),
                   "l2": "no flush: one step's 32 distinct A,B,C sets (2.1 GB) exceed the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "pct_tensor_peak": round(achieved / tensor_peak, 4) if tensor_peak else None,
        "per_scheduler": {k: {kk: vv for kk, vv in v.items() if kk != "per_k_ms"} for k, v in per_sched.items()},
        "persistent_ahead_at_every_K": (all(min(s_, c_) < n_ for s_, c_, n_ in zip(
            per_sched["static"]["per_k_ms"], per_sched["clc"]["per_k_ms"], per_sched["nonpersistent"]["per_k_ms"]))
            if all(k in per_sched for k in SCHED_NAMES) else None),
        "per_k_roofline": per_k_roof,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * len(problems),
        "clocks": clocks,
        "peaks": {"tensor_tflops": tensor_peak, "tensor_tflops_sustained": tensor_peak_sus, "hbm_gbs": hbm,
                  "source": peaks_src},
    }
    if extra is not None:
        line["square_8192_bf16"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(problems, xs)
    return line


def device_inputs(p, seed):
    """Seeded inputs of problem p generated on the GPU (timing-only extras;
    the tests check parity on these shapes with CPU-generated inputs)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    if p.dtype == wl.E4M3:
        a = torch.randn(p.M, p.K, device="cuda", generator=g)
        b = torch.randn(p.N, p.K, device="cuda", generator=g)
        sa, sb = 448.0 / float(a.abs().max()), 448.0 / float(b.abs().max())
        out = ((a * sa).clamp(-448, 448).to(torch.float8_e4m3fn), (b * sb).clamp(-448, 448).to(torch.float8_e4m3fn),
               sa, sb)
        torch.cuda.synchronize()   # drawn on the default stream; the GEMMs run on others
        return out
    td = torch.float16 if p.dtype == wl.F16 else torch.bfloat16
    s = 1.0 / math.sqrt(p.K)
    out = ((torch.randn(p.M, p.K, device="cuda", generator=g) * s).to(td),
           (torch.randn(p.N, p.K, device="cuda", generator=g) * s).to(td), 1.0, 1.0)
    torch.cuda.synchronize()   # drawn on the default stream; the GEMMs run on others
    return out


def time_one(pts, h, p, A, B, C, sa, sb, sched, stream, reps):
    for _ in range(2):
        pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, sa, sb, stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for r in range(reps):
            pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, sched, sa, sb, stream)
            ev[r + 1].record(stream)
    torch.cuda.synchronize()
    if pts.gemm_check(h, stream)[0] != 0:
        raise RuntimeError(f"device error in {p.name}")
    return statistics.median(ev[r].elapsed_time(ev[r + 1]) for r in range(reps))


def extra_configs(pts, dev, stream):
    """The other workloads, TFLOP/s per scheduler: e4m3 8192^3, the tail
    shapes, two GEMMs at once on two streams, the half-occupied GPU and the
    grouped launches."""
    out = {}
    h = pts.gemm_create(dev, pts.make_opts(cta_group=0))
    try:
        probs = wl.e4m3_8192() + wl.bf16_tail()
        for i, p in enumerate(probs):
            A, B, sa, sb = device_inputs(p, 7000 + i)
            C = torch.empty(p.M, p.N, dtype=wl.output_torch_dtype(p.dtype), device="cuda")
            reps = 5 if p.M * p.N * p.K > 2 ** 38 else 10
            row = {}
            for si, name in enumerate(SCHED_NAMES):
                ms = time_one(pts, h, p, A, B, C, sa, sb, si, stream, reps)
                row[name] = round(gemm_flops(p.M, p.N, p.K) / (ms * 1e-3) / 1e12, 1)
            out[p.name] = row
            del A, B, C
        # two GEMMs in flight at once on two streams: the case CLC redistributes work for
        pa, pb = wl.bf16_tail()[0], wl.bf16_tail()[2]
        ins = [device_inputs(pa, 7100), device_inputs(pb, 7101)]
        Cs = [torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda") for p in (pa, pb)]
        hs = [h, pts.gemm_create(dev, pts.make_opts(cta_group=0))]
        streams = [stream, torch.cuda.Stream()]
        conc = {}
        try:
            for si, name in enumerate(SCHED_NAMES):
                times = []
                for rep in range(6):
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(streams[0])
                    streams[1].wait_event(e0)
                    for hh, s_, p, (A, B, sa, sb), C in zip(hs, streams, (pa, pb), ins, Cs):
                        pts.gemm_run(hh, p.M, p.N, p.K, A, B, C, p.dtype, si, sa, sb, s_)
                    end1 = torch.cuda.Event()
                    end1.record(streams[1])
                    streams[0].wait_event(end1)
                    e1.record(streams[0])
                    torch.cuda.synchronize()
                    if rep >= 2:
                        times.append(e0.elapsed_time(e1))
                for hh, s_ in zip(hs, streams):
                    if pts.gemm_check(hh, s_)[0] != 0:
                        raise RuntimeError("device error in the concurrent pair")
                ms = statistics.median(times)
                conc[name] = {"ms": round(ms, 4), "tflops": round(
                    (gemm_flops(pa.M, pa.N, pa.K) + gemm_flops(pb.M, pb.N, pb.K)) / (ms * 1e-3) / 1e12, 1)}
        finally:
            pts.gemm_destroy(hs[1])
        out["concurrent_" + pa.name + "+" + pb.name] = conc
        out["half_occupied"] = half_occupied(pts, dev, stream)
        out["bf16_grouped_vark"] = grouped_vark(pts, dev, stream)
        out["fp16_4096_ksweep_one_grouped_launch"] = sweep_as_grouped(pts, dev, stream)
        out["fp16_4096_tile_plans"] = tile_plans_small_k(pts, dev, stream)
    finally:
        pts.gemm_destroy(h)
    out["note"] = ("library's CTA group per GEMM (pairs from 14 k-blocks per tile for the persistent "
                   "schedulers, from 64 for the non-persistent grid); median of back-to-back "
                   "launches; inputs generated on the GPU from seeded generators (parity for these shapes is in "
                   "the tests)")
    return out


def tile_plans_small_k(pts, dev, stream, ks=(128, 256, 512, 1024), n=20, nbuf=4):
    """The fp16 4096^2 sweep's small-K end under each tile plan the library
    has: the wide 128x256 tile as single CTAs and as CTA pairs (256x256), the
    narrow 128x128 tile as single CTAs (two per SM) and as CTA pairs (256x128,
    one CTA per SM), and the library's own choice.  Per scheduler, microseconds
    per launch over `n` chained launches on `nbuf` rotating buffer sets; whole
    tiles (no stream-K share, no tail halves) in the fixed plans, so that they
    differ in the tile alone."""
    plans = {"wide_cg1": dict(cta_group=1, tile_n=256, split=1, split_k=-1),
             "wide_cg2": dict(cta_group=2, tile_n=256, split=1, split_k=-1),
             "narrow_cg1": dict(cta_group=1, tile_n=128),
             "narrow_cg2": dict(cta_group=2, tile_n=128),
             "library": {}}
    out = {"K": list(ks)}
    for name in plans:
        out[name] = {sn: [] for sn in SCHED_NAMES}
    for K in ks:
        p = wl.fp16_4096_ksweep([K])[0]
        ins = [device_inputs(p, 9500 + 10 * K + i) for i in range(nbuf)]
        Cs = [torch.empty(p.M, p.N, dtype=torch.float16, device="cuda") for _ in range(nbuf)]
        for name, kw in plans.items():
            h = pts.gemm_create(dev, pts.make_opts(**kw))
            try:
                for si, sn in enumerate(SCHED_NAMES):
                    def run(i):
                        A, B, _, _ = ins[i % nbuf]
                        pts.gemm_run(h, p.M, p.N, p.K, A, B, Cs[i % nbuf], p.dtype, si, 1.0, 1.0, stream)
                    for i in range(3):
                        run(i)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for i in range(n):
                        run(i)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if pts.gemm_check(h, stream)[0] != 0:
                        raise RuntimeError(f"device error in the tile-plan sweep ({name}, K={K})")
                    out[name][sn].append(round(e0.elapsed_time(e1) / n * 1e3, 2))
            finally:
                pts.gemm_destroy(h)
        del ins, Cs
    out["note"] = (f"microseconds per launch, {n} chained launches on {nbuf} rotating buffer sets; "
                   "wide = 128x256 per CTA, narrow = 128x128 per CTA; cg2 = CTA pairs; the fixed plans run "
                   "whole tiles, library = the library's own plan")
    return out


def half_occupied(pts, dev, stream, reps=6):
    """SM availability that differs from the static assumption: a long GEMM
    (one 128x256 tile per CTA on half the SMs, K=32768, about 0.2 ms) starts
    first on one stream, then the measured GEMM (5120x5120x4096) on another.
    A static grid sized to the whole GPU leaves half of its CTAs, and their
    tiles, waiting for the occupier to finish; CLC lets the resident CTAs take
    those tiles over."""
    half = torch.cuda.get_device_properties(dev).multi_processor_count // 2
    occ = wl.Problem(f"occupier_{half * 128}x256x32768", half * 128, 256, 32768, wl.BF16, "normal_sqrtk", 7200)
    main = wl.Problem("bf16_5120x5120x4096", 5120, 5120, 4096, wl.BF16, "normal_sqrtk", 7201)
    io = device_inputs(occ, 7200)
    im = device_inputs(main, 7201)
    Co = torch.empty(occ.M, occ.N, dtype=torch.bfloat16, device="cuda")
    Cm = torch.empty(main.M, main.N, dtype=torch.bfloat16, device="cuda")
    ho = pts.gemm_create(dev, pts.make_opts(cta_group=1, split=1))   # one CTA per tile, no slicing
    hm = pts.gemm_create(dev, pts.make_opts(cta_group=1))
    s_occ = torch.cuda.Stream()
    out = {}
    try:
        for si, name in enumerate(SCHED_NAMES):
            times = []
            for rep in range(reps):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s_occ)
                stream.wait_event(e0)
                pts.gemm_run(ho, occ.M, occ.N, occ.K, io[0], io[1], Co, occ.dtype, pts.GEMM_SCHED_STATIC, 1.0, 1.0,
                             s_occ)
                t_launch = time.perf_counter()
                while time.perf_counter() - t_launch < 25e-6:   # let the occupier's CTAs become resident
                    pass
                pts.gemm_run(hm, main.M, main.N, main.K, im[0], im[1], Cm, main.dtype, si, 1.0, 1.0, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if rep >= 2:
                    times.append(e0.elapsed_time(e1))
            if pts.gemm_check(hm, stream)[0] != 0 or pts.gemm_check(ho, s_occ)[0] != 0:
                raise RuntimeError("device error in the half-occupied run")
            out[name] = {"main_done_ms": round(statistics.median(times), 4)}
    finally:
        pts.gemm_destroy(ho)
        pts.gemm_destroy(hm)
    out["note"] = (f"time from the occupier's start ({occ.name}, {half} CTAs, one wave) to the end of the "
                   f"measured GEMM ({main.name}, single CTAs), launched 25 us after the occupier")
    return out


def grouped_vark(pts, dev, stream, reps=10, cgs=(1, 2), scheds=tuple(SCHED_NAMES)):
    """The grouped workload (64 bf16 problems of M=N=1024, K log-uniform in
    [256, 8192]) in ONE launch per scheduler and CTA group: TFLOP/s over all
    problems' flops, median of back-to-back launches (the same problem list
    each time, so the problem table is uploaded once)."""
    probs = wl.bf16_grouped_vark()
    ins = [device_inputs(p, 8000 + i) for i, p in enumerate(probs)]
    Cs = [torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda") for p in probs]
    lst = [(p.M, p.N, p.K, A, B, C) for p, (A, B, _, _), C in zip(probs, ins, Cs)]
    flops = sum(gemm_flops(p.M, p.N, p.K) for p in probs)
    ks = [p.K for p in probs]
    out = {"problems": len(probs), "M": probs[0].M, "N": probs[0].N, "K_min": min(ks), "K_max": max(ks),
           "K_mean": round(sum(ks) / len(ks), 1)}
    arr = pts.gemm.group_array(lst)   # marshalled once: the timed loop makes only the C calls
    for cg in cgs:
        for order, suffix in ((1, ""), (2, "_given_order")):
            h = pts.gemm_create(dev, pts.make_opts(cta_group=cg, group_order=order))
            try:
                for si, name in enumerate(SCHED_NAMES):
                    if name not in scheds:
                        continue
                    for _ in range(3):
                        pts.gemm_run_grouped(h, arr, wl.BF16, si, stream)
                    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
                    with torch.cuda.stream(stream):
                        for r in range(reps):
                            ev[r].record(stream)
                            pts.gemm_run_grouped(h, arr, wl.BF16, si, stream)
                        ev[reps].record(stream)
                    torch.cuda.synchronize()
                    if pts.gemm_check(h, stream)[0] != 0:
                        raise RuntimeError("device error in the grouped run")
                    ms = statistics.median(ev[r].elapsed_time(ev[r + 1]) for r in range(reps))
                    out[f"cg{cg}_{name}{suffix}"] = round(flops / (ms * 1e-3) / 1e12, 1)
            finally:
                pts.gemm_destroy(h)
    h = pts.gemm_create(dev, None)
    try:
        out["auto_cta_group"] = int(pts.gemm_query_grouped(h, lst, wl.BF16, 1).cta_group)
    finally:
        pts.gemm_destroy(h)
    out["note"] = (f"median of {reps} back-to-back grouped launches; TFLOP/s over all {len(probs)} problems; "
                   "problems listed most k-blocks first (the default) or in the given order")
    return out


def sweep_as_grouped(pts, dev, stream, reps=10, rounds=3):
    """The 32 GEMMs of the fp16 K sweep (M = N = 4096, K = 128..4096) as ONE
    grouped launch per scheduler, library defaults: no launch boundary, so no
    per-GEMM start-up, fill and tail (the headline times them as 32 launches,
    as the pages' sweeps do).  The schedulers take turns over `rounds` rounds
    (median over all their launches): this sustained load heats the GPU by
    several percent within a second, which would otherwise penalise whichever
    scheduler is measured last."""
    probs = wl.fp16_4096_ksweep()
    ins = [device_inputs(p, 9000 + i) for i, p in enumerate(probs)]
    Cs = [torch.empty(p.M, p.N, dtype=torch.float16, device="cuda") for p in probs]
    arr = pts.gemm.group_array([(p.M, p.N, p.K, A, B, C) for p, (A, B, _, _), C in zip(probs, ins, Cs)])
    flops = sum(gemm_flops(p.M, p.N, p.K) for p in probs)
    out = {}
    h = pts.gemm_create(dev, None)
    try:
        out["cta_group"] = int(pts.gemm_query_grouped(h, arr, wl.F16, 1).cta_group)
        times = {name: [] for name in SCHED_NAMES}
        per_round = max(1, reps // rounds)
        for _ in range(rounds):
            for si, name in enumerate(SCHED_NAMES):
                for _ in range(3):
                    pts.gemm_run_grouped(h, arr, wl.F16, si, stream)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(per_round + 1)]
                with torch.cuda.stream(stream):
                    for r in range(per_round):
                        ev[r].record(stream)
                        pts.gemm_run_grouped(h, arr, wl.F16, si, stream)
                    ev[per_round].record(stream)
                torch.cuda.synchronize()
                if pts.gemm_check(h, stream)[0] != 0:
                    raise RuntimeError("device error in the grouped sweep")
                times[name] += [ev[r].elapsed_time(ev[r + 1]) for r in range(per_round)]
        for name in SCHED_NAMES:
            out[name] = round(flops / (statistics.median(times[name]) * 1e-3) / 1e12, 1)
    finally:
        pts.gemm_destroy(h)
    out["note"] = (f"median of {rounds} x {per_round} launches per scheduler, the schedulers taking turns each "
                   f"round; TFLOP/s over the 32 GEMMs; most k-blocks first")
    return out


def config_points(pts, dev, stream):
    """One GEMM per configuration point, static scheduler, library defaults,
    each launched twice (a warm-up, then the measured one): fp16 512^3, fp16
    4096^2 x {128, 1024, 4096}, bf16 8192^2 x {1024, 4096, 8192}, e4m3 8192^3
    and the three tail shapes.  For profiling every point with one ncu
    command; prints each point's event time of the second launch."""
    probs = (wl.fp16_512() + wl.fp16_4096_ksweep([128, 1024, 4096]) + wl.bf16_8192_ksweep([1024, 4096, 8192])
             + wl.e4m3_8192() + wl.bf16_tail())
    out = {}
    h = pts.gemm_create(dev, None)
    try:
        for i, p in enumerate(probs):
            A, B, sa, sb = device_inputs(p, 9500 + i)
            C = torch.empty(p.M, p.N, dtype=wl.output_torch_dtype(p.dtype), device="cuda")
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_STATIC, sa, sb, stream)
                ev[0].record(stream)
                pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, pts.GEMM_SCHED_STATIC, sa, sb, stream)
                ev[1].record(stream)
            torch.cuda.synchronize()
            if pts.gemm_check(h, stream)[0] != 0:
                raise RuntimeError(f"device error in {p.name}")
            ms = ev[0].elapsed_time(ev[1])
            out[p.name] = {"us": round(ms * 1e3, 1), "tflops": round(gemm_flops(p.M, p.N, p.K) / (ms * 1e-3) / 1e12, 1),
                           "cta_group": int(pts.gemm_query(h, p.M, p.N, p.K, p.dtype, 1).cta_group)}
            del A, B, C
    finally:
        pts.gemm_destroy(h)
    return out


def square_8192(pts, dev, stream, reps=10, cgs=(1, 2), scheds=tuple(SCHED_NAMES), dtype="bf16", group_m=8):
    """bf16 (or e4m3) 8192^3 per scheduler and CTA group (the >= 70 % of peak target)."""
    p = wl.bf16_8192_ksweep([8192])[0] if dtype == "bf16" else wl.e4m3_8192()[0]
    x = wl.make_inputs(p)
    A, B = x.A.cuda(), x.B.cuda()
    sa, sb = (x.scale_a, x.scale_b) if dtype == "e4m3" else (1.0, 1.0)
    C = torch.empty(p.M, p.N, dtype=torch.bfloat16, device="cuda")
    out = {}
    for cg in cgs:
        h = pts.gemm_create(dev, pts.make_opts(cta_group=cg, group_size_m=group_m))
        try:
            for si, name in enumerate(SCHED_NAMES):
                if name not in scheds:
                    continue
                for _ in range(3):
                    pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, si, sa, sb, stream)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
                with torch.cuda.stream(stream):
                    for r in range(reps):
                        ev[r].record(stream)
                        pts.gemm_run(h, p.M, p.N, p.K, A, B, C, p.dtype, si, sa, sb, stream)
                    ev[reps].record(stream)
                torch.cuda.synchronize()
                if pts.gemm_check(h, stream)[0] != 0:
                    raise RuntimeError("device error in the 8192^3 run")
                ms = statistics.median(ev[r].elapsed_time(ev[r + 1]) for r in range(reps))
                out[f"cg{cg}_{name}"] = round(gemm_flops(p.M, p.N, p.K) / (ms * 1e-3) / 1e12, 1)
        finally:
            pts.gemm_destroy(h)
    ab_mb = (A.numel() * A.element_size() + B.numel() * B.element_size()) / 1e6
    out["note"] = (f"median of {reps} back-to-back launches; A,B = {ab_mb:.0f} MB (L2 is 129 MB); "
                   f"GROUP_SIZE_M {group_m}")
    return out


# ------------------------------------------------------------ reference arm

def run_reference(args, dist, rank, world):
    """The oracle as it stands, on the host cores.  Step s computes rows
    0..R-1 of the sweep's GEMM number s mod 32 (round robin over the K values),
    so any --steps/--warmup finishes in minutes."""
    if rank != 0:
        return None
    from oracle import gemm as og
    problems = wl.fp16_4096_ksweep()
    xs = [wl.make_inputs(p) for p in problems]
    rows = args.ref_rows
    bits = [(x.bits("A").reshape(-1)[: rows * x.problem.K], x.bits("B").reshape(-1)) for x in xs]

    def step(s):
        i = s % len(problems)
        p = problems[i]
        og.gemm(rows, p.N, p.K, bits[i][0], bits[i][1], p.dtype)
        return gemm_flops(rows, p.N, p.K)

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    flops = sum(step(s) for s in range(args.steps))
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    sample = (f"per step rows 0..{rows - 1} ({rows}x4096 outputs, fp64 triple loop) of one sweep GEMM, "
              f"K values taken round robin")
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded inputs as our arm)",
            "config": {"workload": WORKLOAD, "sample": sample}, "impl": "reference",
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": og.max_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--no-square", dest="square", action="store_false")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the other workloads (bf16 8192 sweep points, e4m3, tail shapes, concurrent pair)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--ks", type=int, nargs="*", default=None, help="subset of the sweep's K values")
    ap.add_argument("--scheds", nargs="*", default=SCHED_NAMES, choices=SCHED_NAMES)
    ap.add_argument("--cta-group", type=int, default=0, choices=[0, 1, 2],
                    help="0 = the library's choice per GEMM (single CTAs below 14 k-blocks per tile, "
                         "below 64 for the non-persistent grid)")
    ap.add_argument("--split-k", type=int, default=0, choices=[0, 1, -1],
                    help="stream-K share of the last waves: 0 = the library's choice, 1 = always, -1 = never")
    ap.add_argument("--epilogue", type=int, default=0, choices=[0, 1, 2],
                    help="0 default, 1 TMA stores through shared memory, 2 direct stores from registers")
    ap.add_argument("--graph", action="store_true",
                    help="capture the 32 launches of a step in a CUDA graph and replay it (default: every step "
                         "launches them one by one with gemm_run)")
    ap.add_argument("--square-only", action="store_true",
                    help="only the 8192^3 measurement (for profiling it), restricted by --cta-group, --scheds "
                         "and --square-dtype; prints its numbers, not the benchmark line")
    ap.add_argument("--square-dtype", choices=["bf16", "e4m3"], default="bf16")
    ap.add_argument("--group-size-m", type=int, default=8,
                    help="with --square-only: tile-rows per group of the tile order (the library's default is 8)")
    ap.add_argument("--points", action="store_true",
                    help="only one GEMM per configuration point, twice each (for profiling them); prints their "
                         "times, not the benchmark line")
    ap.add_argument("--grouped-only", action="store_true",
                    help="only the grouped 64-problem measurement (for profiling it), restricted by --cta-group and "
                         "--scheds; prints its numbers, not the benchmark line")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="only time the oracle on whole configuration problems (host cores, about a minute); "
                         "prints those times, not the benchmark line")
    args = ap.parse_args()
    if args.oracle_configs:
        print(json.dumps(oracle_full_configs()), flush=True)
        return
    if args.square_only:
        import persistent_tile_scheduled_gb300 as pts
        pts.load(build_if_missing=False)
        out = square_8192(pts, 0, torch.cuda.Stream(), cgs=(args.cta_group,) if args.cta_group else (1, 2),
                          scheds=tuple(args.scheds), dtype=args.square_dtype, group_m=args.group_size_m)
        print(json.dumps({f"square_8192_{args.square_dtype}": out}), flush=True)
        return
    if args.points:
        import persistent_tile_scheduled_gb300 as pts
        pts.load(build_if_missing=False)
        print(json.dumps({"config_points": config_points(pts, 0, torch.cuda.Stream())}), flush=True)
        return
    if args.grouped_only:
        import persistent_tile_scheduled_gb300 as pts
        pts.load(build_if_missing=False)
        out = grouped_vark(pts, 0, torch.cuda.Stream(), cgs=(args.cta_group,) if args.cta_group else (1, 2),
                           scheds=tuple(args.scheds))
        print(json.dumps({"bf16_grouped_vark": out}), flush=True)
        return
    if args.warmup < 3:
        log("warm-up raised to 3 steps")
        args.warmup = 3
    dist, rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, dist, rank, world)
    else:
        line = run_ours(args, dist, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
