import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) and the CUDA library")


@pytest.fixture(scope="session")
def tq():
    """The C-ABI binding with the CUDA library loaded (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dit_convrot_linear_gb300 import tq as binding
    binding.load()
    return binding
