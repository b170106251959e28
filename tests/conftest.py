import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library through its C ABI)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Print how much of the per-row error bound each labelled parity case
    used (rows that needed the conditioning factor, the largest factor, the
    worst error as a fraction of its bound)."""
    from parity import STATS, format_stats
    if not STATS:
        return
    terminalreporter.write_sep("-", "parity statistics")
    for label, st in STATS:
        terminalreporter.write_line(format_stats(label, st))
