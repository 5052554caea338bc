"""Pins of the oracle's FP8 rounding (the FP8-P variant of forward recipe R2)
against brute force and against torch's float8 casts.

The brute-force side decodes every code of E5M2 and E4M3FN from its bit
layout and picks the nearest value by enumeration, ties to the even code,
saturating at the largest finite value; the oracle uses a closed form in
float64. torch's float8_e5m2 / float8_e4m3fn casts (round to nearest even)
are a second, independent reference inside the finite range. Source: the
FastVideo pull request "Add Attn-QAT training Triton kernels", review of the
FP8 branch (tl.float8e5, Triton's E5M2), and the torch.float8_e4m3fn of the
FastVideo attn_qat_infer page."""
import numpy as np
import pytest
import torch

from oracle import fp8



def decode(fmt):
    """All finite non-negative values of the format, indexed by their code."""
    if fmt == "e5m2":
        vals = []
        for code in range(0x7C):                   # exponent field 31: inf / NaN
            e, m = code >> 2, code & 3
            vals.append(m / 4 * 2.0 ** -14 if e == 0 else (1 + m / 4) * 2.0 ** (e - 15))
        return np.array(vals)
    vals = []
    for code in range(0x7F):                       # 0x7F: NaN
        e, m = code >> 3, code & 7
        vals.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


def nearest_even(a, grid):
    a = np.asarray(a, dtype=np.float64)
    out = np.empty_like(a)
    codes = np.arange(len(grid))
    for i0 in range(0, a.size, 1 << 14):
        x = a.ravel()[i0:i0 + (1 << 14)]
        d = np.abs(x[:, None] - grid[None, :])
        m = d.min(axis=1, keepdims=True)
        cand = d == m
        two = cand.sum(axis=1) == 2
        even = cand & (codes % 2 == 0)[None, :]
        code = np.where(two, np.argmax(even, axis=1), np.argmax(cand, axis=1))
        code = np.where(x > grid[-1], len(grid) - 1, code)
        out.ravel()[i0:i0 + x.size] = grid[code]
    return out


def brute(x, fmt):
    x = np.asarray(x, dtype=np.float64)
    return np.copysign(nearest_even(np.abs(x), decode(fmt)), x)


def all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    return x[np.isfinite(x)].astype(np.float64)


FMTS = ["e5m2", "e4m3"]


@pytest.mark.parametrize("fmt", FMTS)
def test_grid_decodes(fmt):
    g = decode(fmt)
    assert np.all(np.diff(g) > 0)
    assert g[-1] == fp8.FORMATS[fmt][2]
    assert len(g) == (124 if fmt == "e5m2" else 127)
    np.testing.assert_array_equal(fp8.fp8_round(g, fmt), g)        # every code is a fixed point


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_value(fmt):
    x = all_finite_bf16()
    np.testing.assert_array_equal(fp8.fp8_round(x, fmt), brute(x, fmt))


@pytest.mark.parametrize("fmt", FMTS)
def test_midpoints_and_neighbouring_fp32(fmt):
    g = decode(fmt)
    mid = (g[:-1] + g[1:]) / 2                   # every tie (exact in FP32)
    assert np.all(mid.astype(np.float32).astype(np.float64) == mid)
    m32 = mid.astype(np.float32)
    x = np.concatenate([mid, np.nextafter(m32, np.float32(np.inf)).astype(np.float64),
                        np.nextafter(m32, np.float32(0)).astype(np.float64), -mid])
    np.testing.assert_array_equal(fp8.fp8_round(x, fmt), brute(x, fmt))
    # ties go to the even code: the value with an even last mantissa bit
    t = fp8.fp8_round(mid, fmt)
    codes = np.searchsorted(g, t)
    assert np.all(codes % 2 == 0)


@pytest.mark.parametrize("fmt,dtype", [("e5m2", torch.float8_e5m2), ("e4m3", torch.float8_e4m3fn)])
def test_matches_torch_float8_casts(fmt, dtype):
    rng = np.random.default_rng(7)
    vmax = fp8.FORMATS[fmt][2]
    x = np.concatenate([rng.uniform(0, 1, 100000), np.exp(rng.uniform(np.log(1e-9), np.log(vmax), 100000)),
                        -rng.uniform(0, 1, 1000)]).astype(np.float32)
    want = torch.from_numpy(x).to(dtype).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.fp8_round(x.astype(np.float64), fmt), want)


def test_saturation_and_signed_zero():
    assert fp8.fp8_round([1e9], "e5m2")[0] == 57344.0
    assert fp8.fp8_round([1e9], "e4m3")[0] == 448.0
    z = fp8.fp8_round([-1e-30], "e5m2")[0]
    assert z == 0 and np.signbit(z)
