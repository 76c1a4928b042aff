import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The GPU parity cases' near-tie counts and whether their backward
    comparisons ran, one line per case (shown with -q too)."""
    mod = sys.modules.get("tests.parity")
    reports = getattr(mod, "REPORTS", None) if mod is not None else None
    if not reports:
        return
    tr = terminalreporter
    tr.section("parity summary: near-tie tokens and compared outputs per case")
    n_ties = 0
    for case, kw in reports:
        n_ties += int(kw.get("near_tie_tokens", 0))
        tr.write_line(f"{case}: " + ", ".join(f"{k}={v}" for k, v in kw.items()))
    all_bwd = all(kw.get("backward_compared", True) for _, kw in reports)
    tr.write_line(f"{len(reports)} cases, {n_ties} near-tie tokens in total, "
                  f"backward comparisons ran in every case: {all_bwd}")
