"""The debug build (libattnqat_checked.so): its bounds checks count what they
skip, and the attention kernels' parity suites run clean under them.

Every plain global load and store of the attention kernels sits behind a check
that its element index lies inside its buffer's extent; in the debug build a
failing check skips the access and counts it (attnqat_debug_oob_count), so an
indexing bug shows up as a count instead of a fault. This stands in for a
memory checker, which is not available on this GPU pool."""
import ctypes
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_the_checks_count_what_they_skip():
    """In a fresh process on the debug build: of n + extra guarded writes to an
    n-element buffer the last `extra` are skipped and counted, the rest land."""
    code = r'''
import ctypes, sys, torch
sys.path.insert(0, sys.argv[1])
from fp4_quantization_aware_gb300 import attnqat, build
build.build(checked=True)
lib = attnqat.load(attnqat.CHECKED_LIB_PATH)
assert lib.attnqat_checked_build() == 1
n, extra = 1000, 37
buf = torch.full((n + 64,), -1.0, device="cuda")   # 64 canaries past the n elements
cnt = ctypes.c_ulonglong(0)
attnqat.check(lib.attnqat_debug_oob_count(ctypes.byref(cnt), 1), "clear")
attnqat.check(lib.attnqat_selftest_bounds(ctypes.c_void_p(buf.data_ptr()), n, extra, None), "selftest_bounds")
attnqat.check(lib.attnqat_debug_oob_count(ctypes.byref(cnt), 1), "count")
assert cnt.value == extra, cnt.value
h = buf.cpu()
assert torch.equal(h[:n], torch.arange(n, dtype=torch.float32)), "in-bounds writes"
assert bool((h[n:] == -1.0).all()), "a skipped write landed"
attnqat.check(lib.attnqat_debug_oob_count(ctypes.byref(cnt), 0), "count")
assert cnt.value == 0
print("bounds selftest ok")
'''
    r = subprocess.run([sys.executable, "-c", code, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "bounds selftest ok" in r.stdout


def test_parity_suites_run_clean_on_the_debug_build():
    """The small-shape parity suites of every kernel family (QAT forward and
    backward at D = 64 and 128, causal, ragged and cross shapes; recipe R2 in
    all P formats; the inference forward and NVFP4 packing; the abort path) on
    the debug build, each test followed by a check that nothing was skipped."""
    env = dict(os.environ, ATTNQAT_TEST_CHECKED="1")
    sel = "parity_small or outputs_untouched or test_r2_gpu or test_infer_gpu or test_abort_gpu"
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", sel, "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_attn_gpu.py"), os.path.join(ROOT, "tests", "test_r2_gpu.py"),
                        os.path.join(ROOT, "tests", "test_infer_gpu.py"), os.path.join(ROOT, "tests", "test_abort_gpu.py")],
                       capture_output=True, text=True, timeout=1500, cwd=ROOT, env=env)
    tail = r.stdout[-3000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    # the selection covers 74 tests; a rename that drops some must not pass silently
    assert m and int(m.group(1)) >= 70, tail
    assert "failed" not in r.stdout and "skipped" not in r.stdout, tail
