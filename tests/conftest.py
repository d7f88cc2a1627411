import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def ref():
    """The oracle module (built on first use)."""
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library's binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import activation_backward_gb300 as cba
    cba.load()
    return cba
