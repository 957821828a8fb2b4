import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (large oracle passes)")


def have_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The compiled FLCE library on a CUDA device; the GPU tests fail loudly without it."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import linear_cross_entropy_tcgen05_gb300 as flce
    flce.load_library()
    return flce
