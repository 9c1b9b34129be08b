import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The error distribution of the session's parity comparisons, per input
    dtype: the plain normalised metric beside the bounded one (which does not
    charge the output format's own rounding) and per-element percentiles."""
    try:
        from helpers import PARITY_LOG
    except ImportError:
        return
    if not PARITY_LOG:
        return
    import json
    tr = terminalreporter
    tr.section("parity: error distribution (normalised by s * sum_k |a||b|)")
    tr.write_line(f"{'dtype':6} {'cases':>6} {'elements':>11} {'plain max':>11} {'bounded max':>12} "
                  f"{'p50':>10} {'p99':>10} {'p99.9':>10}")
    for dt in sorted({r["dtype"] for r in PARITY_LOG}):
        rs = [r for r in PARITY_LOG if r["dtype"] == dt]
        tr.write_line(f"{dt:6} {len(rs):6d} {sum(r['elements'] for r in rs):11d} "
                      f"{max(r['plain_max'] for r in rs):11.3e} {max(r['bounded_max'] for r in rs):12.3e} "
                      f"{max(r['p50'] for r in rs):10.3e} {max(r['p99'] for r in rs):10.3e} "
                      f"{max(r['p999'] for r in rs):10.3e}")
    path = os.environ.get("PTS_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(PARITY_LOG, f)
