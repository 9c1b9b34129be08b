"""bench.py's output line on a GPU: one short run of our arm, every key the
line promises, and the arithmetic that ties them together (throughput from
the step time, the roofline fraction, the bytes the end-to-end leg moves, the
launches counted)."""
import json
import os
import subprocess
import sys

import pytest
import torch

import workloads as wl

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3", "--no-extras",
           "--no-square"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [s for s in r.stdout.splitlines() if s.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_contract_keys(line):
    import bench
    d = line
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "f16"
    assert d["data"].startswith("synthetic") and "workload" in d["config"]
    assert set(d["per_scheduler"]) == {"nonpersistent", "static", "clc"}
    assert isinstance(d["clocks"]["reasons"], list) and "sm_mhz" in d["clocks"] and "sm_max_mhz" in d["clocks"]


def test_value_from_step_time(line):
    flops = sum(2 * p.M * p.N * p.K for p in wl.fp16_4096_ksweep())
    d = line
    assert d["value"] > 0
    assert d["value"] == pytest.approx(flops / (d["ms_per_step"] * 1e-3) / 1e12, rel=1e-3)
    assert d["value"] == pytest.approx(d["per_scheduler"]["static"]["value"], abs=0.01)   # the line rounds to 0.01


def test_roofline_block(line):
    r = line["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(line["value"], rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-3)
    assert r["traffic"] is None or r["traffic"] > 0
    # a short run (3 steps) is compared with the burst peak
    peaks = line["peaks"]
    assert r["peak"] == peaks["tensor_tflops"] and "burst" in r["peak_source"]
    assert r["frac_burst"] == pytest.approx(r["frac"], rel=1e-3)
    assert r["frac_sustained"] == pytest.approx(r["achieved"] / peaks["tensor_tflops_sustained"], rel=1e-3)


def test_end_to_end_leg_counts_its_bytes(line):
    e = line["e2e"]
    probs = wl.fp16_4096_ksweep()
    assert e["value"] > 0 and e["unit"] == "TFLOP/s"
    assert e["h2d_bytes_per_step"] == sum(2 * (p.M + p.N) * p.K for p in probs)   # A and B, fp16
    assert e["d2h_bytes_per_step"] == sum(2 * p.M * p.N for p in probs)           # C, fp16
    assert e["value"] < line["value"]


def test_launches_and_cpu_baseline(line):
    assert line["gpu_launches"] == 32 * line["steps"]
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["unit"] == "TFLOP/s"
    assert "whole GEMMs" in c["sample"]
