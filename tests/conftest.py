import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work (full-size oracle runs)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library on a GPU machine (builds it if needed)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_quantization_aware_gb300 import attnqat
    from fp4_quantization_aware_gb300 import build as builder
    builder.build()
    return attnqat.load()
