import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Per-comparison parity records of the GPU tests (tests/gpu_helpers.py):
    rows compared, rows with an element above the plain bound, largest errors."""
    try:
        from gpu_helpers import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.section("parity records")
    tr.write_line(f"{'test':<78} {'rows':>9} {'>tol':>6} {'max|dO|':>9} {'max|dLSE|':>10} {'oracle_s':>8}")
    for r in PARITY_LOG:
        os_ = "" if r.get("oracle_s") is None else f"{r['oracle_s']:.1f}"
        tr.write_line(f"{r['test'][-78:]:<78} {r['rows']:>9} {r['rows_above_plain_tol']:>6} "
                      f"{r['max_err_o']:>9.2e} {r['max_err_lse']:>10.2e} {os_:>8}")
    out = os.environ.get("BSP_PARITY_LOG")
    if out:
        with open(out, "w") as f:
            json.dump(PARITY_LOG, f, indent=1)
