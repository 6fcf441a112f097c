import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "fullsize: a GPU parity case at a full benchmark size (slow oracle)")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (built in-tree first if missing or stale)."""
    from linear_cross_entropy_tmem_gb300 import binding
    from linear_cross_entropy_tmem_gb300.build import build
    build()
    return binding.load()
