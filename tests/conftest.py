import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (built in-tree by __graft_entry__.build())."""
    from varlen_sliding_window_gb300 import binding
    return binding.load_library()
