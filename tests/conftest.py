import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library through its Python binding; fails loudly when missing."""
    if not has_gpu():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    import broadcast_target_attention_gb300 as ikbo
    ikbo.load()
    return ikbo
