"""Pins of the oracle's NVFP4 fake quantizer against brute force and worked groups.

The brute-force side decodes the E4M3FN and E2M1 formats from their bit
layouts, picks the nearest grid value by enumeration with an even-code
tie-break, and divides in native float32; the oracle uses closed forms in
float64. Sources: "NVFP4 Attention QAT Backward" (cuDNN frontend docs,
Overview) and the Attn-QAT paper summary (Method: E2M1, group size 16).
"""
import os

import numpy as np
import pytest

from oracle import nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked.txt")


# ---------------------------------------------------------------- brute force
def e4m3fn_values():
    """All finite non-negative E4M3FN values, indexed by their 7-bit code."""
    vals = []
    for code in range(0x7F):          # 0x7F is NaN in E4M3FN
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def e2m1_values():
    vals = []
    for code in range(8):
        e, m = code >> 1, code & 1
        vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    return np.array(vals)


def nearest_even(a, grid):
    """Nearest grid value to each non-negative a; ties go to the even code.

    Values above the grid's maximum saturate to it (satfinite)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.empty_like(a)
    codes = np.arange(len(grid))
    for i0 in range(0, a.size, 1 << 16):
        x = a.ravel()[i0:i0 + (1 << 16)]
        d = np.abs(x[:, None] - grid[None, :])
        m = d.min(axis=1, keepdims=True)
        cand = d == m
        two = cand.sum(axis=1) == 2
        even = cand & (codes % 2 == 0)[None, :]
        code = np.where(two, np.argmax(even, axis=1), np.argmax(cand, axis=1))
        code = np.where(x > grid[-1], len(grid) - 1, code)
        out.ravel()[i0:i0 + x.size] = grid[code]
    return out


E4 = e4m3fn_values()
E2 = e2m1_values()


def brute_group(x):
    """Fake-quantize one group with native float32 division and enumeration."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32))
    s = nearest_even(np.float32(amax) / np.float32(6.0), E4)[()]
    if s == 0:
        return np.copysign(np.zeros(len(x32)), x32)
    q = x32 / np.float32(s)                     # IEEE float32 division
    e = nearest_even(np.abs(q.astype(np.float64)), E2)
    return np.copysign(e * s, x32)


def all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    return x[np.isfinite(x)].astype(np.float64)


# ---------------------------------------------------------------- pins
def test_grids_decode():
    assert len(E4) == 127 and E4.max() == 448.0 and E4[1] == 2.0 ** -9
    assert list(E2) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_rounding_exhaustive_points():
    mids = (E4[1:] + E4[:-1]) / 2
    pts = np.concatenate([E4, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                          np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.abs(all_finite_bf16()),
                          np.random.default_rng(0).uniform(0, 600, 20000).astype(np.float32),
                          np.random.default_rng(1).uniform(0, 0.02, 20000).astype(np.float32)])
    pts = nvfp4.fl32(pts)
    np.testing.assert_array_equal(nvfp4.rne_e4m3(pts), nearest_even(pts, E4))


def test_e4m3_scale_of_every_bf16_amax():
    amax = np.abs(all_finite_bf16())
    s32 = (amax.astype(np.float32) / np.float32(6.0)).astype(np.float64)
    np.testing.assert_array_equal(nvfp4.group_scale(amax), nearest_even(s32, E4))


def test_e4m3_amax_on_ties():
    mids = (E4[1:] + E4[:-1]) / 2            # exact: at most 5 significant bits
    amax = 6.0 * mids                         # exact, and amax/6 == mid exactly
    got = nvfp4.group_scale(amax)
    codes = np.searchsorted(E4, got)
    assert np.all(E4[codes] == got)
    assert np.all(codes % 2 == 0)             # every tie went to the even code


def test_e2m1_rounding_points():
    mids = (E2[1:] + E2[:-1]) / 2
    m32 = mids.astype(np.float32)
    pts = np.concatenate([E2, mids, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0)),
                          [6.5, 7.0, 100.0, 1e30],
                          np.random.default_rng(2).uniform(0, 7, 50000).astype(np.float32)]).astype(np.float64)
    np.testing.assert_array_equal(nvfp4.rne_e2m1(pts), nearest_even(pts, E2))
    np.testing.assert_array_equal(nvfp4.rne_e2m1(-pts), -nearest_even(pts, E2))
    assert np.signbit(nvfp4.rne_e2m1(np.array([-0.1])))[0]


@pytest.mark.parametrize("chunk", range(4))
def test_element_step_every_bf16_times_every_scale(chunk):
    """fl32(x/s) then E2M1 RNE, for all finite BF16 x and all nonzero E4M3 s."""
    x = all_finite_bf16()
    ax = np.abs(x).astype(np.float32)
    for s in E4[1:][chunk::4]:
        got = nvfp4.quantize_with_scale(x, s)
        with np.errstate(over="ignore"):
            q = (ax / np.float32(s)).astype(np.float64)   # native float32 division
        want = np.copysign(nearest_even(q, E2) * s, x)
        np.testing.assert_array_equal(got.view(np.int64), want.view(np.int64))


def test_element_step_near_midpoints_fp32():
    """FP32 inputs one ulp either side of every exact midpoint m*s."""
    mids = (E2[1:] + E2[:-1]) / 2
    for s in E4[1:]:
        t = (mids * s).astype(np.float32)
        x = np.concatenate([t, np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(0))])
        got = nvfp4.quantize_with_scale(x.astype(np.float64), s)
        want = nearest_even((x / np.float32(s)).astype(np.float64), E2) * s
        np.testing.assert_array_equal(got, want)


def test_groups_against_brute_force():
    rng = np.random.default_rng(3)
    groups = []
    for mag in (1e-4, 1e-3, 6e-3, 0.05, 1.0, 30.0, 3000.0, 1e5):
        groups.append((rng.standard_normal((300, 16)) * mag).astype(np.float32))
    groups.append(rng.uniform(0, 0.02, (500, 16)).astype(np.float32))   # probability-like
    g = np.concatenate(groups).astype(np.float64)
    got = nvfp4.fake_nvfp4(g, axis=1)
    want = np.stack([brute_group(row) for row in g])
    np.testing.assert_array_equal(got.view(np.int64), want.view(np.int64))


def test_ragged_axis_and_orientation():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 37)).astype(np.float32).astype(np.float64)
    got = nvfp4.fake_nvfp4(x, axis=1)
    for r in range(3):
        for g0 in range(0, 37, 16):
            seg = x[r, g0:g0 + 16]
            np.testing.assert_array_equal(got[r, g0:g0 + 16], brute_group(seg))
    np.testing.assert_array_equal(nvfp4.fake_nvfp4(x.T, axis=0), got.T)


def test_sign_symmetry_and_bf16_exactness():
    x = np.random.default_rng(5).standard_normal((64, 128)).astype(np.float32).astype(np.float64) * 3
    y = nvfp4.fake_nvfp4(x)
    np.testing.assert_array_equal(nvfp4.fake_nvfp4(-x).view(np.int64), (-y).view(np.int64))
    y32 = y.astype(np.float32)
    assert np.all((y32.view(np.uint32) & 0xFFFF) == 0)   # every output is a BF16 value


def _parse(tok):
    out = []
    for t in tok.split():
        v, _, n = t.partition("*")
        out += [float(v)] * (int(n) if n else 1)
    return np.array(out)


def test_worked_groups():
    n = 0
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        name, xs, s, ys = (p.strip() for p in line.split("|"))
        x, want = _parse(xs), _parse(ys)
        assert nvfp4.group_scale(np.max(np.abs(x)))[()] == float(s), name
        got = nvfp4.fake_nvfp4(x)
        np.testing.assert_array_equal(got.view(np.int64), want.view(np.int64), err_msg=name)
        n += 1
    assert n == 5


def test_device_zero_scale_threshold_is_exact():
    """The kernels skip the quantizer for groups with amax <= kZeroScaleAmax;
    that constant must be exactly the largest FP32 amax whose scale is zero."""
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "fp4_quantization_aware_gb300", "csrc", "nvfp4.cuh")).read()
    t = np.float32(float(re.search(r"kZeroScaleAmax = ([0-9.e+-]+)f", src).group(1)))
    up = np.nextafter(t, np.float32(1))
    assert nvfp4.group_scale(np.float64(t)) == 0.0
    assert nvfp4.group_scale(np.float64(up)) > 0.0
    assert nearest_even(np.float64(t / np.float32(6)), E4)[()] == 0.0
    assert nearest_even(np.float64(up / np.float32(6)), E4)[()] > 0.0
