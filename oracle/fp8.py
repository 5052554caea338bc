"""FP8 rounding of probabilities for the FP8-P variant of forward recipe R2:
the oracle.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The library's CUDA
path never calls it, and it shares no code with that path.

Source: the FastVideo pull request "Add Attn-QAT training Triton kernels",
review of the one-pass forward's FP8 branch ("when dtype is tl.float8e5
(FP8) ..."): the probabilities of a key tile are cast to an FP8 type before
the P V product, and the row sum is taken from the unquantized P. The
review names Triton's ``tl.float8e5``, the E5M2 format; E4M3FN (the
``torch.float8_e4m3fn`` of the FastVideo attn_qat_infer page) is offered as
the other FP8 type. The cast of an FP32 value is round to nearest, ties to
the even code:

* E5M2: 2 mantissa bits, exponent bias 15, normal values 1.mm * 2^e for e in
  [-14, 15] (largest finite 1.75 * 2^15 = 57344), subnormals multiples of
  2^-16 below 2^-14.
* E4M3FN: 3 mantissa bits, bias 7, normal e in [-6, 8] (largest finite 448),
  subnormals multiples of 2^-9, no infinities.

Values beyond the largest finite one saturate to it (probabilities of the
recipe never exceed 1, so the choice does not arise there). Signs are kept.

Parity pins (tests/test_oracle_fp8.py): enumeration of every code of both
formats decoded from its bit layout, nearest value with even-code ties, on
every finite BF16 value and on FP32 values around every midpoint; and
torch's own float8 casts on FP32 values inside the finite range.
"""
from __future__ import annotations

import numpy as np

FORMATS = {
    # name: (mantissa bits, smallest normal exponent, largest finite)
    "e5m2": (2, -14, 57344.0),
    "e4m3": (3, -6, 448.0),
}


def fp8_round(x, fmt: str) -> np.ndarray:
    """Round float64 values (FP32-exact in use) to the FP8 format ``fmt``
    ("e5m2" or "e4m3"), ties to the even code, saturating; float64 out."""
    mbits, emin, vmax = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    out = np.zeros_like(a)
    min_normal = 2.0 ** emin
    sub = a < min_normal
    step_sub = 2.0 ** (emin - mbits)               # subnormal spacing
    out[sub] = np.rint(a[sub] / step_sub) * step_sub
    nrm = ~sub
    if np.any(nrm):
        _, e = np.frexp(a[nrm])                    # a = f * 2^e, f in [0.5, 1)
        step = np.ldexp(1.0, e - 1 - mbits)        # mbits bits below the leading 1
        out[nrm] = np.minimum(np.rint(a[nrm] / step) * step, vmax)
    return np.copysign(out, x)
