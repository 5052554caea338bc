"""ctypes binding of libattnqat (the C ABI in include/attnqat.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels. PyTorch provides device memory and streams. There is
no fallback: ``load()`` raises if the library has not been built, and every
non-OK status becomes an ``AttnQatError``.

The raw entry points are available with their C names on the loaded library
(``load().attnqat_fwd(...)``); the functions below wrap them for torch tensors.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattnqat.so")
# the debug build: bounds checks on every plain global access, counted
# (attnqat_debug_oob_count); for tests, loaded with load(CHECKED_LIB_PATH)
CHECKED_LIB_PATH = os.path.join(HERE, "libattnqat_checked.so")

ATTNQAT_OK = 0
# probability quantizers of recipe R2 (attnqat_p_format)
P_FORMATS = {"nvfp4": 0, "e5m2": 1, "e4m3": 2}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "misaligned", 4: "workspace", 5: "cuda",
          6: "timeout"}


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Sq", ctypes.c_int64), ("Sk", ctypes.c_int64),
                ("D", ctypes.c_int64), ("is_causal", ctypes.c_int32), ("softmax_scale", ctypes.c_float)]


class AttnQatError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status}) {detail}".strip())
        self.status = status


_P = ctypes.c_void_p
_S = ctypes.c_int
_PP = ctypes.POINTER(Problem)
SIGNATURES = {
    "attnqat_version": (ctypes.c_int, []),
    "attnqat_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attnqat_last_error_message": (ctypes.c_char_p, []),
    "attnqat_check_support": (_S, [_PP]),
    "attnqat_fwd_workspace_bytes": (ctypes.c_size_t, [_PP]),
    "attnqat_bwd_workspace_bytes": (ctypes.c_size_t, [_PP]),
    "attnqat_fake_nvfp4": (_S, [_P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "attnqat_fake_nvfp4_f32": (_S, [_P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "attnqat_fwd": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_bwd": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_quantize_qkv": (_S, [_PP, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_fwd_main": (_S, [_PP, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_bwd_preprocess": (_S, [_PP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_bwd_main": (_S, [_PP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_bwd_dq_convert": (_S, [_PP, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_bwd_noalloc": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "attnqat_bwd_host_workspace_bytes": (ctypes.c_size_t, [_PP, ctypes.c_int]),
    "attnqat_bwd_host": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "attnqat_device_status": (_S, [ctypes.c_int]),
    "attnqat_selftest_wait_timeout": (_S, [ctypes.c_uint64, _P]),
    "attnqat_selftest_set_wait_limit": (_S, [ctypes.c_uint64]),
    "attnqat_selftest_quotient": (_S, [_P, _P]),
    "attnqat_selftest_scale": (_S, [_P, _P]),
    "attnqat_nvfp4_pack": (_S, [_P, _P, _P, ctypes.c_int64, ctypes.c_int64, _P]),
    "attnqat_infer_fwd_workspace_bytes": (ctypes.c_size_t, [_PP]),
    "attnqat_infer_fwd_packed": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, _P]),
    "attnqat_infer_fwd": (_S, [_PP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_fwd_r2": (_S, [_PP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_fwd_main_r2": (_S, [_PP, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "attnqat_fwd_r2_p": (_S, [_PP, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "attnqat_fwd_main_r2_p": (_S, [_PP, _P, _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "attnqat_checked_build": (ctypes.c_int, []),
    "attnqat_debug_oob_count": (_S, [ctypes.POINTER(ctypes.c_ulonglong), ctypes.c_int]),
    "attnqat_selftest_bounds": (_S, [_P, ctypes.c_int64, ctypes.c_int64, _P]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Open the built library (raises if it is missing) and declare signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m fp4_quantization_aware_gb300.build` "
                           "(or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    if status != ATTNQAT_OK:
        detail = load().attnqat_last_error_message().decode()
        raise AttnQatError(status, where, detail)


def problem(B, H, Sq, Sk, D, causal=False, scale=None) -> Problem:
    return Problem(B, H, Sq, Sk, D, 1 if causal else 0, 1.0 / math.sqrt(D) if scale is None else scale)


# ------------------------------------------------------------------ torch helpers
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _problem_of(q, k, causal, scale) -> Problem:
    B, H, Sq, D = q.shape
    return problem(B, H, Sq, k.shape[2], D, causal, scale)


def _bf16_contig(*ts):
    import torch
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("tensors must be contiguous CUDA bfloat16 (BHSD)")


def fake_nvfp4(x, stream=None):
    """fake_nvfp4 along the last axis (groups of 16) of a BF16 or FP32 CUDA tensor."""
    import torch
    x = x.contiguous()
    y = torch.empty_like(x)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    lib = load()
    if x.dtype == torch.bfloat16:
        check(lib.attnqat_fake_nvfp4(_ptr(x), _ptr(y), rows, cols, _stream(stream)), "attnqat_fake_nvfp4")
    elif x.dtype == torch.float32:
        check(lib.attnqat_fake_nvfp4_f32(_ptr(x), _ptr(y), rows, cols, _stream(stream)), "attnqat_fake_nvfp4_f32")
    else:
        raise ValueError("fake_nvfp4 takes bfloat16 or float32")
    return y


def workspace(nbytes: int, device):
    import torch
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def fwd(q, k, v, causal=False, scale=None, ws=None, out=None, stream=None):
    """Forward: returns (O, O', LSE) for BHSD BF16 CUDA tensors."""
    import torch
    _bf16_contig(q, k, v)
    p = _problem_of(q, k, causal, scale)
    lib = load()
    need = lib.attnqat_fwd_workspace_bytes(ctypes.byref(p))
    if need == 0:
        check(lib.attnqat_check_support(ctypes.byref(p)), "attnqat_check_support")
    if ws is None:
        ws = workspace(need, q.device)
    if out is None:
        o, o_hp = torch.empty_like(q), torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    else:
        o, o_hp, lse = out
    check(lib.attnqat_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_hp), _ptr(lse), _ptr(ws),
                          ws.numel(), _stream(stream)), "attnqat_fwd")
    return o, o_hp, lse


def fwd_r2(q, k, v, causal=False, scale=None, ws=None, out=None, stream=None, p_format="nvfp4"):
    """Forward in recipe R2 (each key tile's P quantized before normalisation):
    returns (O, O', LSE) for BHSD BF16 CUDA tensors; O' and LSE are those of
    ``fwd``, so ``bwd`` applies unchanged. ``p_format``: "nvfp4" (fake_nvfp4
    of 16-key groups), or "e5m2" / "e4m3" for the FP8-P variant."""
    import torch
    _bf16_contig(q, k, v)
    p = _problem_of(q, k, causal, scale)
    lib = load()
    need = lib.attnqat_fwd_workspace_bytes(ctypes.byref(p))
    if need == 0:
        check(lib.attnqat_check_support(ctypes.byref(p)), "attnqat_check_support")
    if ws is None:
        ws = workspace(need, q.device)
    if out is None:
        o, o_hp = torch.empty_like(q), torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    else:
        o, o_hp, lse = out
    check(lib.attnqat_fwd_r2_p(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_hp), _ptr(lse),
                               P_FORMATS[p_format], _ptr(ws), ws.numel(), _stream(stream)), "attnqat_fwd_r2_p")
    return o, o_hp, lse


def bwd(do, q, k, v, o_hp, lse, causal=False, scale=None, ws=None, out=None, stream=None):
    """Backward: returns (dQ, dK, dV) for BHSD BF16 CUDA tensors."""
    import torch
    _bf16_contig(do, q, k, v, o_hp)
    p = _problem_of(q, k, causal, scale)
    lib = load()
    need = lib.attnqat_bwd_workspace_bytes(ctypes.byref(p))
    if need == 0:
        check(lib.attnqat_check_support(ctypes.byref(p)), "attnqat_check_support")
    if ws is None:
        ws = workspace(need, q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    check(lib.attnqat_bwd(ctypes.byref(p), _ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(o_hp), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)), "attnqat_bwd")
    return dq, dk, dv


def nvfp4_pack(x, stream=None):
    """Real NVFP4 encoding along the last axis (a multiple of 16) of a BF16 CUDA
    tensor: (packed uint8 (..., n/2), scales uint8 E4M3 (..., n/16))."""
    import torch
    _bf16_contig(x)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    packed = torch.empty(*x.shape[:-1], cols // 2, dtype=torch.uint8, device=x.device)
    scales = torch.empty(*x.shape[:-1], cols // 16, dtype=torch.uint8, device=x.device)
    lib = load()
    check(lib.attnqat_nvfp4_pack(_ptr(x), _ptr(packed), _ptr(scales), rows, cols, _stream(stream)),
          "attnqat_nvfp4_pack")
    return packed, scales


def infer_fwd(q, k, v, causal=False, scale=None, ws=None, out=None, with_lse=True, stream=None):
    """Inference forward with NVFP4 Q, K and BF16 V: returns (O, LSE or None)."""
    import torch
    _bf16_contig(q, k, v)
    p = _problem_of(q, k, causal, scale)
    lib = load()
    need = lib.attnqat_infer_fwd_workspace_bytes(ctypes.byref(p))
    if need == 0:
        check(lib.attnqat_check_support(ctypes.byref(p)), "attnqat_check_support")
        raise AttnQatError(2, "attnqat_infer_fwd", "the inference forward needs D == 128")
    if ws is None:
        ws = workspace(need, q.device)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device) if with_lse else None
    else:
        o, lse = out
    check(lib.attnqat_infer_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(ws),
                                ws.numel(), _stream(stream)), "attnqat_infer_fwd")
    return o, lse


def infer_fwd_packed(q_fp4, q_sf, k_fp4, k_sf, v, causal=False, scale=None, out=None, with_lse=True,
                     stream=None):
    """Inference forward on pre-packed NVFP4 Q, K (``nvfp4_pack`` output, BHS
    leading axes) and BF16 V: returns (O, LSE or None)."""
    import torch
    B, H, Sq, _ = q_fp4.shape
    D = v.shape[3]
    p = problem(B, H, Sq, k_fp4.shape[2], D, causal, scale)
    if out is None:
        o = torch.empty(B, H, Sq, D, dtype=torch.bfloat16, device=v.device)
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=v.device) if with_lse else None
    else:
        o, lse = out
    check(load().attnqat_infer_fwd_packed(ctypes.byref(p), _ptr(q_fp4), _ptr(q_sf), _ptr(k_fp4), _ptr(k_sf),
                                          _ptr(v), _ptr(o), _ptr(lse), _stream(stream)),
          "attnqat_infer_fwd_packed")
    return o, lse


def device_status(clear: bool = True) -> int:
    """The device error word (0 = ok, 6 = a bounded wait timed out); synchronizes."""
    return load().attnqat_device_status(1 if clear else 0)


def _autograd_function():
    import torch

    class AttnQatFunction(torch.autograd.Function):
        """O = fake_nvfp4(P) V^ in the forward; the QAT backward (dQ, dK from the
        unquantized P, dV = fake_nvfp4(P)^T dO) from the saved O' and LSE."""

        @staticmethod
        def forward(ctx, q, k, v, causal, scale):
            q, k, v = (t.contiguous() for t in (q, k, v))
            o, o_hp, lse = fwd(q, k, v, causal=causal, scale=scale)
            ctx.save_for_backward(q, k, v, o_hp, lse)
            ctx.causal, ctx.scale = causal, scale
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o_hp, lse = ctx.saved_tensors
            dq, dk, dv = bwd(do.contiguous(), q, k, v, o_hp, lse, causal=ctx.causal, scale=ctx.scale)
            return dq, dk, dv, None, None

    return AttnQatFunction


_FN = None


def attention(q, k, v, causal: bool = False, scale: Optional[float] = None):
    """Attn-QAT attention for training: BHSD BF16 CUDA tensors in, O out, with
    the QAT backward wired into autograd."""
    global _FN
    if _FN is None:
        _FN = _autograd_function()
    return _FN.apply(q, k, v, causal, 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale)
