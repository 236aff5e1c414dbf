import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library binding; fails loudly when it is missing on a GPU machine."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_linear_gb300 as bl
    return bl
