import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its Python binding (GPU tests only)."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    import switch_top_expert_router_b300 as sm
    sm.load_library()   # raises if the CUDA library is missing
    return sm
