import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity table of the GPU comparisons that ran: the plain max |o - oracle|
    (no allowance for the output's own bf16 rounding) beside the tolerance."""
    helpers = sys.modules.get("gpu_helpers")
    log = getattr(helpers, "PARITY_LOG", None)
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity vs the oracle: %d comparisons" % len(log))
    by_test = {}
    for test, what, dt, tol, err, used, lerr in log:
        key = (test.split("::")[0].split("/")[-1], dt, tol)
        cur = by_test.setdefault(key, [0, 0.0, 0.0, 0.0])
        cur[0] += 1
        cur[1] = max(cur[1], err)
        cur[2] = max(cur[2], used)
        cur[3] = max(cur[3], lerr or 0.0)
    tr.write_line("%-28s %-9s %8s %6s %14s %14s %12s" % (
        "file", "dtype", "tol_o", "n", "max|o-oracle|", "tol share used", "max|lse err|"))
    for (f, dt, tol), (n, err, used, lerr) in sorted(by_test.items()):
        tr.write_line("%-28s %-9s %8.0e %6d %14.3e %14.2f %12.3e" % (f, dt, tol, n, err, used,
                                                                      lerr))
