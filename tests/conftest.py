import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the compiled library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The parity errors of this run, one line per (test, tensor): relative L2 error and the largest
    element error over max|reference| (the normwise reading of the 2e-3 target)."""
    try:
        import _parity
    except ImportError:
        return
    if not _parity.REPORT:
        return
    tr = terminalreporter
    tr.section("parity against the oracle (rel L2, max elem / max|ref|)")
    worst = {}
    for test, name, rel, elem in _parity.REPORT:
        tr.write_line(f"{test:<90s} {name:<4s} {rel:.3e} {elem:.3e}")
        w = worst.get(name, (0.0, 0.0))
        worst[name] = (max(w[0], rel), max(w[1], elem))
    for name, (rel, elem) in sorted(worst.items()):
        tr.write_line(f"worst {name:<4s} rel L2 {rel:.3e}  max elem {elem:.3e}")
