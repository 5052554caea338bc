"""The C-ABI library builds, loads and exports every declared symbol; its
host-side validation answers without touching a GPU."""
import ctypes
import math
import os
import re

import pytest

from fp4_quantization_aware_gb300 import attnqat
from fp4_quantization_aware_gb300 import build as builder

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attnqat.h")


@pytest.fixture(scope="module")
def clib():
    builder.build()
    return attnqat.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attnqat_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(clib):
    names = declared_functions()
    assert len(names) >= 15
    raw = ctypes.CDLL(attnqat.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    assert set(names) == set(attnqat.SIGNATURES), "binding and header disagree"


def test_debug_build_exports_the_same_symbols_and_says_so(clib):
    builder.build(checked=True)
    raw = ctypes.CDLL(attnqat.CHECKED_LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing
    raw.attnqat_checked_build.restype = ctypes.c_int
    assert raw.attnqat_checked_build() == 1
    assert clib.attnqat_checked_build() == 0


def test_product_build_has_no_bounds_checks(clib):
    n = ctypes.c_ulonglong(7)
    assert clib.attnqat_debug_oob_count(ctypes.byref(n), 0) == 2            # unsupported
    assert clib.attnqat_selftest_bounds(None, 16, 4, None) == 2             # nothing launched
    assert b"debug build" in clib.attnqat_last_error_message()


def test_version_and_status_strings(clib):
    assert clib.attnqat_version() >= 100
    assert clib.attnqat_status_string(0) == b"ok"
    assert clib.attnqat_status_string(6) == b"device wait timed out"
    assert clib.attnqat_status_string(99) == b"unknown status"


def _support(clib, **kw):
    p = attnqat.problem(**{**dict(B=1, H=2, Sq=256, Sk=256, D=64), **kw})
    return clib.attnqat_check_support(ctypes.byref(p))


def test_check_support(clib):
    assert _support(clib) == 0
    assert _support(clib, D=128, Sq=32760, Sk=32760) == 0
    assert _support(clib, Sq=100, Sk=300) == 0                       # non-causal cross attention
    assert _support(clib, D=96) == 2
    assert _support(clib, causal=True, Sq=100, Sk=300) == 2
    assert _support(clib, Sq=0) == 1
    assert _support(clib, B=300, H=300) == 2
    assert _support(clib, B=1 << 62, H=4) == 2                       # B*H wraps to 0 in 64 bits: still rejected
    assert _support(clib, B=1, H=65535) == 0 and _support(clib, B=1, H=65536) == 2
    assert _support(clib, Sq=(1 << 31) - 256, Sk=100) == 2           # sequence lengths past the kernels' int range
    assert _support(clib, scale=float("nan")) == 1
    assert _support(clib, scale=-1.0) == 1
    assert clib.attnqat_check_support(None) == 1
    assert b"head dimension" in clib.attnqat_last_error_message() or True


def test_workspace_sizes(clib):
    p = attnqat.problem(1, 16, 4096, 4096, 128)
    bh = 16
    fwd = clib.attnqat_fwd_workspace_bytes(ctypes.byref(p))
    bwd = clib.attnqat_bwd_workspace_bytes(ctypes.byref(p))
    # Q^, K^, V^ (BF16) and, at D = 128, the split-tile area of pass 2 (128
    # counter words and, for min(query tiles, 96) tiles, both CTAs' FP32 [O', O]
    # slots) and NVFP4 Q and K (E2M1 pairs + E4M3 scales)
    fsplit = 128 * 4 + min(bh * 4096 // 128, 96) * 2 * 2 * 128 * 128 * 4
    assert fwd == 3 * bh * 4096 * 128 * 2 + fsplit + 2 * (bh * 4096 * 64 + bh * 4096 * 8)
    base = 3 * bh * 4096 * 128 * 2
    # + delta, the FP32 dQ accumulator, the split-tile area (128 counter words
    # and FP32 [dK, dV] slots for min(key tiles, 96) tiles) and, at D = 128,
    # the NVFP4 Q and K of the backward's S recompute
    split = 128 * 4 + min(bh * 4096 // 128, 96) * 2 * 128 * 128 * 4
    packed = 2 * (bh * 4096 * 64 + bh * 4096 * 8)
    assert bwd == base + bh * 4096 * 4 + bh * 4096 * 128 * 4 + split + packed
    small = attnqat.problem(1, 1, 100, 300, 64)      # 3 key tiles of 64-wide rows
    assert clib.attnqat_bwd_workspace_bytes(ctypes.byref(small)) == (
        256 * ((100 * 64 * 2 + 255) // 256) + 2 * 256 * ((300 * 64 * 2 + 255) // 256)
        + 256 * ((100 * 4 + 255) // 256) + 256 * ((100 * 64 * 4 + 255) // 256)
        + 256 * ((128 * 4 + 3 * 2 * 128 * 64 * 4 + 255) // 256))
    bad = attnqat.problem(1, 1, 10, 10, 96)
    assert clib.attnqat_fwd_workspace_bytes(ctypes.byref(bad)) == 0


def test_host_backward_workspace_sizes(clib):
    """attnqat_bwd_host needs two head-group slots: each group's dO, Q, O',
    K, V, LSE, dQ, dK, dV and its attnqat_bwd workspace (256-byte rounded)."""
    p = attnqat.problem(1, 16, 4096, 4096, 128)
    r = lambda x: (x + 255) // 256 * 256
    g = attnqat.problem(1, 4, 4096, 4096, 128)          # 16 heads in 4 groups of 4
    tile = 4 * 4096 * 128 * 2
    slot = 8 * r(tile) + r(4 * 4096 * 4) + r(clib.attnqat_bwd_workspace_bytes(ctypes.byref(g)))
    assert clib.attnqat_bwd_host_workspace_bytes(ctypes.byref(p), 4) == 2 * slot
    # chunks are clamped to 1 .. B*H; unsupported problems give 0
    one = attnqat.problem(1, 1, 4096, 4096, 128)
    slot1 = 8 * r(tile // 4) + r(4096 * 4) + r(clib.attnqat_bwd_workspace_bytes(ctypes.byref(one)))
    assert clib.attnqat_bwd_host_workspace_bytes(ctypes.byref(p), 100) == 2 * slot1
    assert clib.attnqat_bwd_host_workspace_bytes(ctypes.byref(p), 0) == clib.attnqat_bwd_host_workspace_bytes(
        ctypes.byref(p), 1)
    bad = attnqat.problem(1, 1, 10, 10, 96)
    assert clib.attnqat_bwd_host_workspace_bytes(ctypes.byref(bad), 2) == 0


def test_errors_before_any_launch(clib):
    p = attnqat.problem(1, 1, 128, 128, 64)
    buf = ctypes.create_string_buffer(1 << 20)
    a = ctypes.addressof(buf)
    base = (a + 255) & ~255
    # null tensor
    st = clib.attnqat_fwd(ctypes.byref(p), None, base, base, base, base, base, base, 1 << 19, None)
    assert st == 1
    # misaligned tensor
    st = clib.attnqat_fwd(ctypes.byref(p), base + 2, base, base, base, base, base, base, 1 << 19, None)
    assert st == 3
    # workspace too small
    st = clib.attnqat_fwd(ctypes.byref(p), base, base, base, base, base, base, base, 16, None)
    assert st == 4
    assert b"needs" in clib.attnqat_last_error_message()
    # unsupported head dim
    bad = attnqat.problem(1, 1, 128, 128, 80)
    st = clib.attnqat_bwd(ctypes.byref(bad), base, base, base, base, base, base, base, base, base, base, 1 << 19, None)
    assert st == 2
    # quantizer: negative size, null pointers
    assert clib.attnqat_fake_nvfp4(base, base, -1, 16, None) == 1
    assert clib.attnqat_fake_nvfp4(None, base, 4, 16, None) == 1
    assert clib.attnqat_fake_nvfp4_f32(base, base, 0, 16, None) == 0       # empty: nothing to do


def test_binding_raises_with_detail(clib):
    with pytest.raises(attnqat.AttnQatError) as e:
        attnqat.check(3, "x")
    assert e.value.status == 3


def test_problem_default_scale():
    p = attnqat.problem(1, 1, 8, 8, 128)
    assert math.isclose(p.softmax_scale, 1 / math.sqrt(128), rel_tol=1e-7)
