import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (CPU-side checks only need it to load)."""
    from exact_io_aware_107_b300 import _binding
    return _binding.load()
