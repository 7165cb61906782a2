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
def ops():
    """The library binding, built if needed. Skips without a CUDA device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_hadamard_rotated_gb300 import build, ops as _ops
    build.build()
    _ops.lib()
    return _ops
