import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the session's parity counts (GEMM tolerance, SwiGLU blocks)."""
    try:
        from helpers import parity_lines
    except ImportError:
        return
    lines = parity_lines()
    if lines:
        terminalreporter.write_sep("-", "parity counts per test")
        for line in lines:
            terminalreporter.write_line(line)
