"""bench.py's host-side rules (no GPU): which tensor peak a run's roofline
fraction is taken against."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_short_runs_take_the_burst_peak_and_long_ones_the_sustained():
    burst, sus = 1943.5, 1725.2
    assert bench.roofline_peak(0.029, burst, sus) == (burst, False)      # 20 steps of the sweep
    assert bench.roofline_peak(0.329, burst, sus) == (sus, True)         # 200 steps
    assert bench.roofline_peak(bench.LONG_RUN_S, burst, sus) == (sus, True)
    assert bench.roofline_peak(5.0, burst, None) == (burst, False)      # no sustained figure known
