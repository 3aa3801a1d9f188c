import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The CUDA library's Python binding, built in-tree; GPU tests only."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import selective_state_space_ssm_gb300 as ssm
    ssm.load()
    return ssm
