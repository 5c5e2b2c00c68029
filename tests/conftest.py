import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """Plain max relative error of every float output the GPU parity tests compared (over
    entries with |ref| >= 1e-3 * magnitude), next to the tolerance."""
    from helpers import REL_ERR
    if not REL_ERR:
        return
    tr = terminalreporter
    tr.section("max relative error per test and output (|ref| >= 1e-3 * magnitude)")
    for (test, what), (err, n, tol) in sorted(REL_ERR.items()):
        tr.write_line(f"max_rel_err {err:.3e} tol {tol:.0e} n {n} {test} :: {what}")
