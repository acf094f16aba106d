import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_terminal_summary(terminalreporter):
    """Report the plain maximum relative error of every float parity
    comparison (elements with |oracle| >= 1e-3 rms), next to the floored
    metric the tests assert."""
    try:
        from helpers import PLAIN_REPORT
    except ImportError:
        return
    if not PLAIN_REPORT:
        return
    worst = {}
    for case, qty, v in PLAIN_REPORT:
        key = (qty, case)
        worst[key] = max(worst.get(key, 0.0), v)
    terminalreporter.section("plain max relative error over |oracle| >= 1e-3 rms")
    for (qty, case), v in sorted(worst.items()):
        terminalreporter.write_line("%-14s %-40s %.3e" % (qty, case, v))
