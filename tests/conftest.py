import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library, or skip when no GPU is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sliding_window_attention_02_gb300 as rswa
    rswa.load()  # raises if the shared library is missing
    return rswa
