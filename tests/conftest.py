import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU work (full-size oracle runs)")


# ATTNQAT_TEST_CHECKED=1 runs the GPU tests against the debug build
# (libattnqat_checked.so), whose bounds checks skip and count any plain global
# access outside its buffer; every test then also requires a count of zero.
CHECKED = os.environ.get("ATTNQAT_TEST_CHECKED") == "1"


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library on a GPU machine (builds it if needed)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp4_quantization_aware_gb300 import attnqat
    from fp4_quantization_aware_gb300 import build as builder
    builder.build(checked=CHECKED)
    lib = attnqat.load(attnqat.CHECKED_LIB_PATH if CHECKED else attnqat.LIB_PATH)
    assert lib.attnqat_checked_build() == (1 if CHECKED else 0)
    return lib


@pytest.fixture(autouse=True)
def _no_skipped_access(request):
    """Debug build only: no test may make a kernel skip an access."""
    yield
    if CHECKED and "lib" in request.fixturenames:
        import ctypes
        lib = request.getfixturevalue("lib")
        n = ctypes.c_ulonglong(0)
        assert lib.attnqat_debug_oob_count(ctypes.byref(n), 1) == 0
        assert n.value == 0, f"{n.value} accesses outside their buffers were skipped"
