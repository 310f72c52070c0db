import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA binding; skips cleanly where no GPU is visible."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_moe_expert_router_gb300 as moe
    moe.load()
    return moe
