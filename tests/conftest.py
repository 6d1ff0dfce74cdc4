import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def zblib():
    """Builds (if needed) and loads libzb; CPU-only calls work without a GPU."""
    from backward_split_linear_gb300 import _build, binding

    _build.build()
    return binding.lib()


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from backward_split_linear_gb300 import _build, binding

    _build.build()
    binding.lib()
    return torch.device("cuda:0")
