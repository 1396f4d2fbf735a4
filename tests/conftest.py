import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


@pytest.fixture(scope="session")
def augtree_lib():
    """The C-ABI library, built in-tree first if it is missing or older than its sources."""
    from shared_prompt_tree_gb300 import build
    build.build()
    import shared_prompt_tree_gb300 as at
    return at.lib()


@pytest.fixture(scope="session")
def cuda_device(augtree_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    torch.cuda.set_device(0)
    return torch.device("cuda", 0)
