import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_terminal_summary(terminalreporter):
    """Near ties counted by the GPU parity tests (decisions within 1e-6 of a
    threshold, in uniform units, which are excused from the bit-exact
    comparison): one line per case."""
    try:
        import parity
    except ImportError:
        return
    rows = getattr(parity, "NEAR_TIES", [])
    if not rows:
        return
    agg = {}
    for case, near, n in rows:
        a = agg.setdefault(case, [0, 0])
        a[0] += near
        a[1] += n
    terminalreporter.write_sep("-", "near ties (excused from bit-exact comparison)")
    for case, (near, n) in sorted(agg.items()):
        terminalreporter.write_line("%-60s %4d of %6d requests" % (case, near, n))
