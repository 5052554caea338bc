"""CPU float64 oracle of Attn-QAT (NVFP4 fake-quantized attention).

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. It shares no code with
the CUDA path in ``fp4_quantization_aware_gb300``, and neither imports the
other.
"""
from .fp8 import fp8_round  # noqa: F401
from .nvfp4 import fake_nvfp4, fl32, group_scale, quantize_with_scale, rne_e2m1, rne_e4m3  # noqa: F401
from .attn import (attn_qat_bwd, attn_qat_fwd, bwd_head, dkdv_keys, dq_rows, fwd_head, fwd_rows,  # noqa: F401
                   hats, infer_fwd, lse_ohp_head, nvfp4_codes, p_hat, probs, r2_fwd, r2_rows, R2_BLOCK_N, R2_P_FORMATS)
