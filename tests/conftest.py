import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu on a GB300)")
    config.addinivalue_line("markers", "slow: full-size problem; takes tens of seconds")


@pytest.fixture(scope="session")
def cuda_device():
    """GPU tests run only where a GPU is expected: a missing device is a failure, not a skip."""
    import torch
    assert torch.cuda.is_available(), "this test needs a CUDA device"
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def pa():
    """The CUDA library's Python binding; fails loudly if the extension is not built."""
    import paged_kv_cache_work_gb300 as m
    m.load()
    return m
