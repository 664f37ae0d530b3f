"""pytest configuration: the ``gpu`` marker and shared fixtures.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything else runs
on the CPU. Run ``pytest -m "not gpu"`` without a GPU.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: long-running case (full-size shapes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The loaded C-ABI library; GPU tests fail (not skip) if it cannot be loaded."""
    from moe_decode_weight_gb300 import api
    return api.lib()
