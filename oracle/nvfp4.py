"""NVFP4 fake quantizer: the oracle.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The library's CUDA
path never calls it, and it shares no code with that path.

Definition followed ("NVFP4 Attention QAT Backward", cuDNN frontend docs,
section *Overview*): values are fake-quantized to the NVFP4 E2M1 format with an
E4M3 scale for every 16 values and immediately dequantized; the local-scale
conversion uses precise division, so exact E2M1 midpoints keep
round-to-nearest-even. The Attn-QAT paper summary (section *Method*) fixes
E2M1 with group size 16.

Per group of 16 values x (read as FP32 numbers):

1. ``amax = max |x_i|`` (exact).
2. ``s32 = fl32(amax / 6)``: one correctly rounded FP32 division.
3. ``s = RNE_E4M3FN(s32)``: nearest E4M3FN value (max 448, subnormal step
   2^-9, no infinities), ties to the even mantissa code, values beyond 448
   saturate to 448.
4. ``s == 0``: every output is a zero carrying the sign of x.
5. otherwise ``q_i = fl32(x_i / s)`` (correctly rounded FP32 division),
   ``e_i = RNE_E2M1(q_i)`` on {0, .5, 1, 1.5, 2, 3, 4, 6} with ties to the
   even code and |q| > 6 saturating to 6, sign kept (so -0 survives), and
   ``y_i = e_i * s`` (exact: at most 6 significant bits, so exactly a BF16).

FP32 operations are emulated by computing in float64 and rounding once to
float32; for one division of two FP32 operands this double rounding is
innocuous because 53 >= 2*24 + 2.

Groups start at index 0 of the quantized axis; a ragged last group is padded
with zeros, which change no amax.

Parity pins: exhaustive brute-force enumeration of the E4M3FN and E2M1 grids
(tests/test_oracle_nvfp4.py) and hand-derived worked groups.
"""
from __future__ import annotations

import numpy as np

GROUP = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUB_STEP = 2.0 ** -9


def fl32(x) -> np.ndarray:
    """Round float64 values to the nearest float32 (ties to even); float64 out.

    Values beyond the float32 range become +-inf, as an FP32 operation would."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def rne_e4m3(v) -> np.ndarray:
    """Round non-negative values to E4M3FN, ties to even, saturating at 448.

    E4M3FN has 3 mantissa bits and exponent bias 7: normal values are
    1.mmm * 2^e for e in [-6, 8] (largest finite 1.75 * 2^8 = 448), and
    subnormals are multiples of 2^-9 below 2^-6.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    sub = v < E4M3_MIN_NORMAL
    out[sub] = np.rint(v[sub] / E4M3_SUB_STEP) * E4M3_SUB_STEP
    nrm = ~sub
    if np.any(nrm):
        _, e = np.frexp(v[nrm])           # v = m * 2^e, m in [0.5, 1)
        step = np.ldexp(1.0, e - 4)       # 3 mantissa bits below the leading 1
        out[nrm] = np.minimum(np.rint(v[nrm] / step) * step, E4M3_MAX)
    return out


def rne_e2m1(q) -> np.ndarray:
    """Round values to the signed E2M1 grid, ties to the even code, saturating.

    E2M1 magnitudes are 0, 0.5, 1, 1.5 (step 0.5 below 2), 2, 3 (step 1 in
    [2, 4)) and 4, 6 (step 2 from 4); within each binade the even code is the
    even multiple of the step, so rounding to the step with rint gives the
    ties-to-even-code result.
    """
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.rint(a / step) * step, E2M1_MAX)
    return np.copysign(r, q)


def group_scale(amax) -> np.ndarray:
    """E4M3 block scale of a group from its amax: RNE_E4M3(fl32(amax / 6))."""
    return rne_e4m3(fl32(np.asarray(amax, dtype=np.float64) / 6.0))


def quantize_with_scale(x, s) -> np.ndarray:
    """Fake-quantize values x with an already chosen E4M3 scale s (broadcast)."""
    x = np.asarray(x, dtype=np.float64)
    s = np.broadcast_to(np.asarray(s, dtype=np.float64), x.shape)
    zero = s == 0.0
    safe = np.where(zero, 1.0, s)
    y = rne_e2m1(fl32(x / safe)) * safe
    return np.where(zero, np.copysign(0.0, x), np.copysign(np.abs(y), x))


def fake_nvfp4(x, axis: int = -1) -> np.ndarray:
    """Fake-quantize x in groups of 16 along ``axis`` (float64 in, float64 out).

    ``x`` must hold FP32-representable values (BF16 activations or FP32
    probabilities). The output values are exactly representable in BF16.
    """
    x = np.asarray(x, dtype=np.float64)
    xm = np.moveaxis(x, axis, -1)
    n = xm.shape[-1]
    pad = (-n) % GROUP
    if pad:
        xm = np.concatenate([xm, np.zeros(xm.shape[:-1] + (pad,))], axis=-1)
    g = xm.reshape(xm.shape[:-1] + (xm.shape[-1] // GROUP, GROUP))
    s = group_scale(np.max(np.abs(g), axis=-1))[..., None]
    y = quantize_with_scale(g, s).reshape(xm.shape)[..., :n]
    return np.moveaxis(y, -1, axis)


def group_scales(x, axis: int = -1) -> np.ndarray:
    """The E4M3 scale of every 16-group along ``axis`` (diagnostics)."""
    xm = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    pad = (-xm.shape[-1]) % GROUP
    if pad:
        xm = np.concatenate([xm, np.zeros(xm.shape[:-1] + (pad,))], axis=-1)
    g = xm.reshape(xm.shape[:-1] + (xm.shape[-1] // GROUP, GROUP))
    return group_scale(np.max(np.abs(g), axis=-1))
