import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
    import __graft_entry__ as g

    g.build_host()


@pytest.fixture(scope="session")
def cuda_built():
    import __graft_entry__ as g

    g.build_cuda()
    return True


@pytest.fixture(scope="session")
def gpu(cuda_built):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test requested but no CUDA device is visible")
    return torch.device("cuda:0")
