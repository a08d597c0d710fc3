import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of host time)")


def has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu_lib():
    """The loaded C-ABI library (GPU tests only). Fails loudly if the extension was not built."""
    if not has_gpu():
        pytest.fail("gpu-marked test run without a visible CUDA device")
    from top_routing_dispatch_moe_gb300 import moe
    return moe
