import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")

# whole-tensor errors of the full-size workloads, printed after the run
_PARITY = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    have_gpu = False
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        pass
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def parity_report():
    """case -> {elements, max_abs_out, max_abs_lse, tol}, filled by the GPU
    parity tests and printed at the end of the session."""
    return _PARITY


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not _PARITY:
        return
    tr = terminalreporter
    tr.section("whole-tensor parity against the oracle (max |GPU - oracle|)")
    for case, r in _PARITY.items():
        tr.write_line(f"{case:18s} {r['elements']:>12d} elements  out {r['max_abs_out']:.3e} "
                      f"(tol {r['tol'][0]:.0e})  lse {r['max_abs_lse']:.3e} (tol {r['tol'][1]:.0e})")


def read_golden(name):
    """Rows of a '|'-separated golden file, comments stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows
