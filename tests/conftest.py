import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if needed (no GPU required to load it)."""
    from head_attention_backward_gb300 import build as _build
    _build.build_library()
    from head_attention_backward_gb300 import binding
    return binding.load()
