import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of CPU time")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its C ABI (built in-tree if missing)."""
    from top_gradient_compression_gb300 import _lib
    return _lib.load()
