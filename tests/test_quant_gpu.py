"""The CUDA fake quantizer is bit-exact to the oracle on identical inputs.

The BF16 path (Q, K, V) and the FP32 path (the routine the attention kernels
apply to P) are compared bit for bit, signed zeros included."""
import numpy as np
import pytest

from fp4_quantization_aware_gb300 import attnqat
from oracle import nvfp4
from parity import to_dev

pytestmark = pytest.mark.gpu


def _bits32(a):
    return np.asarray(a, np.float32).view(np.uint32)


def _gpu(x32, dtype):
    import torch
    t = to_dev(x32.astype(np.float32), dtype)
    y = attnqat.fake_nvfp4(t)
    torch.cuda.synchronize()
    return y.float().cpu().numpy()


def test_bf16_every_pattern(lib):
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(0)
    groups = [x[rng.permutation(x.size)][: x.size // 16 * 16]]               # mixed magnitudes
    groups.append(np.sort(x)[: x.size // 16 * 16])                           # similar magnitudes
    for g in groups:
        g = g.reshape(-1, 16)
        got = _gpu(g, torch.bfloat16)
        want = nvfp4.fake_nvfp4(g.astype(np.float64), axis=1).astype(np.float32)
        np.testing.assert_array_equal(_bits32(got), _bits32(want))


def test_bf16_attention_shapes(lib):
    import torch
    rng = np.random.default_rng(1)
    for D in (64, 128):
        x = (rng.standard_normal((3, 5, 77, D)) * rng.choice([1e-3, 1, 50], (3, 5, 77, 1))).astype(np.float32)
        x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
        got = _gpu(x, torch.bfloat16)
        want = nvfp4.fake_nvfp4(x.astype(np.float64), axis=-1).astype(np.float32)
        np.testing.assert_array_equal(_bits32(got), _bits32(want))


def _e4m3_positive():
    v = []
    for code in range(1, 0x7F):
        e, m = code >> 3, code & 7
        v.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(v)


def test_f32_scale_and_midpoint_edges(lib):
    """Groups whose amax pins every E4M3 scale, with members on every E2M1
    midpoint m*s and one FP32 ulp either side, plus amax on E4M3 ties."""
    import torch
    rows = []
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    for s in _e4m3_positive():
        t = (mids * s).astype(np.float32)
        members = np.concatenate([t, np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(0))])
        for k in range(0, members.size, 15):
            m = members[k:k + 15]
            row = np.zeros(16, np.float32)
            row[0] = np.float32(6.0 * s)               # amax/6 == s exactly
            row[1:1 + m.size] = m
            rows.append(row)
    e4 = np.concatenate([[0.0], _e4m3_positive()])
    for lo, hi in zip(e4[:-1], e4[1:]):                # amax/6 on an E4M3 tie and next to it
        mid = np.float32(6.0 * (lo + hi) / 2)
        for a in (mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))):
            row = np.linspace(0, 1, 16, dtype=np.float32) * a
            rows.append(row.astype(np.float32))
    x = np.stack(rows)
    got = _gpu(x, torch.float32)
    want = nvfp4.fake_nvfp4(x.astype(np.float64), axis=1).astype(np.float32)
    np.testing.assert_array_equal(_bits32(got), _bits32(want))


def test_f32_probability_like(lib):
    import torch
    rng = np.random.default_rng(2)
    p = [rng.exponential(1e-3, (20000, 16)), rng.exponential(1e-2, (20000, 16)),
         rng.uniform(0, 1, (20000, 16)), rng.standard_normal((20000, 16)) * 100]
    x = np.concatenate(p).astype(np.float32)
    got = _gpu(x, torch.float32)
    want = nvfp4.fake_nvfp4(x.astype(np.float64), axis=1).astype(np.float32)
    np.testing.assert_array_equal(_bits32(got), _bits32(want))


@pytest.mark.parametrize("cols", [1, 15, 17, 37, 4096 + 9])
def test_ragged_columns(lib, cols):
    import torch
    x = np.random.default_rng(cols).standard_normal((9, cols)).astype(np.float32)
    for dtype in (torch.float32, torch.bfloat16):
        xr = torch.from_numpy(x).to(dtype).float().numpy()
        got = _gpu(xr, dtype)
        want = nvfp4.fake_nvfp4(xr.astype(np.float64), axis=1).astype(np.float32)
        np.testing.assert_array_equal(_bits32(got), _bits32(want))


def test_in_place(lib):
    import torch
    x = np.random.default_rng(3).standard_normal((64, 128)).astype(np.float32)
    t = to_dev(x, torch.bfloat16)
    ref = attnqat.fake_nvfp4(t).clone()
    lib.attnqat_fake_nvfp4(t.data_ptr(), t.data_ptr(), 64, 128, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(t, ref)


def test_quotient_matches_ieee_division_exhaustively(lib):
    """The quantizer divides by the group scale without a division instruction;
    on every E4M3 scale and every FP32 numerator whose quotient can reach an
    E2M1 decision, the result equals IEEE division bit for bit."""
    import torch
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    attnqat.check(lib.attnqat_selftest_quotient(out.data_ptr(), torch.cuda.current_stream().cuda_stream),
                  "selftest_quotient")
    torch.cuda.synchronize()
    n, a_bits, s_bits = out.cpu().tolist()
    assert n == 0, f"{n} mismatches, e.g. a bits {a_bits & 0xFFFFFFFF:#x}, s bits {s_bits:#x}"


def test_scale_arithmetic_and_nonneg_variant_exhaustively(lib):
    """amax / 6 by FMA correction equals IEEE division for every FP32 amax that
    reaches it; the refined reciprocal equals IEEE reciprocal on every E4M3
    scale; the attention kernels' variant for probabilities equals the generic
    quantizer bit for bit."""
    import torch
    out = torch.zeros(6, dtype=torch.int64, device="cuda")
    attnqat.check(lib.attnqat_selftest_scale(out.data_ptr(), torch.cuda.current_stream().cuda_stream),
                  "selftest_scale")
    torch.cuda.synchronize()
    n_div, n_rcp, n_quant, e_div, e_rcp, e_quant = out.cpu().tolist()
    assert n_div == 0, f"{n_div} amax / 6 mismatches, e.g. amax bits {e_div & 0xFFFFFFFF:#x}"
    assert n_rcp == 0, f"{n_rcp} reciprocal mismatches, e.g. scale bits {e_rcp & 0xFFFFFFFF:#x}"
    assert n_quant == 0, f"{n_quant} group mismatches, e.g. group {e_quant & 0xFFFFFFFFFF}"
