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
