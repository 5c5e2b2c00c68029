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
    """Error statistics of every float output the GPU parity tests compared, one line per
    test function and output: the R17 ratio max |gpu - ref| / max(|ref|, m) that the
    tolerance bounds (m: the oracle's magnitude of the expression), and the plain max
    relative error over entries with |ref| >= 1e-3 m and over those with |ref| >= m / 2."""
    from helpers import REL_ERR
    if not REL_ERR:
        return
    agg = {}
    for (test, what), (ratio, rel, rel2, n, tol) in REL_ERR.items():
        key = (test.split("[")[0].split("::")[-1], what, tol)
        a = agg.setdefault(key, [0.0, 0.0, 0.0, 0, 0])
        agg[key] = [max(a[0], ratio), max(a[1], rel), max(a[2], rel2), a[3] + n, a[4] + 1]
    tr = terminalreporter
    tr.section("parity error per test function and output")
    tr.write_line("R17-ratio (asserted < tol) | plain rel |ref|>=1e-3m | plain rel |ref|>=m/2 | tol | cases | entries | test :: output")
    for (test, what, tol), (ratio, rel, rel2, n, cases) in sorted(agg.items()):
        tr.write_line(f"{ratio:.2e} | {rel:.2e} | {rel2:.2e} | {tol:.0e} | {cases} | {n} | {test} :: {what}")
