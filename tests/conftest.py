import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes on the host)")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library through its Python binding (built in-tree if missing)."""
    from packed_varlen_non_gb300 import build, h3attn
    build.ensure_built()
    return h3attn


# Full-output parity figures (max / mean abs error over every element), printed
# in the terminal summary so that they show even in a quiet run.
_PARITY_LINES = []


@pytest.fixture
def parity_report():
    return _PARITY_LINES.append


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if _PARITY_LINES:
        terminalreporter.write_sep("-", "full-output parity against the fp64 oracle")
        for line in _PARITY_LINES:
            terminalreporter.write_line(line)
