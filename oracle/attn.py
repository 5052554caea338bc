"""Attn-QAT forward and backward: the oracle (float64, CPU, row-blocked).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The library's CUDA
path never calls it, and it shares no code with that path.

Equations ("NVFP4 Attention QAT Backward", cuDNN frontend docs, *Overview*):

    Q^, K^, V^ = fake_nvfp4(Q), fake_nvfp4(K), fake_nvfp4(V)   (groups along D)
    P  = softmax(scale * Q^ K^T)
    O' = P V^                                   (high-precision auxiliary output)
    dS = P * (dO V^T - rowsum(O' * dO))
    dQ = scale * dS K^
    dK = scale * dS^T Q^
    dV = fake_nvfp4(P)^T dO                     (groups of 16 keys)

and the low-precision forward output of the Attn-QAT paper summary (*Method*):
``O = fake_nvfp4(P) V^``. The LSE statistic is the natural-log log-sum-exp of
the scaled logits (cuDNN page, *High-level wrapper*), and the backward
recomputes P from it (paper summary, Fix 2). Causal masking drops keys j > i
(self-attention only, cuDNN page *Current support and limitations*).

Inputs are float64 arrays holding BF16-exact values (and an FP32 LSE in the
backward). P is rounded once to FP32 before it is fake-quantized, because the
quantizer's definition takes FP32 operands. Outputs are float64 and unrounded;
tests round O, O' to BF16 and LSE to FP32 where the CUDA path stores them so.

Parity pins (tests/test_oracle_attn.py): torch SDPA in float64 with the
quantizer set to identity; central finite differences of the STE surrogate
for dQ and dK; linearity in V^ for dV; the FlashAttention identity
rowsum(P * dO V^T) = rowsum(O' * dO); the causal first row in closed form;
a pure-Python brute force on a tiny ragged case.
"""
from __future__ import annotations

import numpy as np

from .fp8 import fp8_round
from .nvfp4 import fake_nvfp4, fl32

ROW_BLOCK = 256


def _identity(x, axis=-1):
    return np.asarray(x, dtype=np.float64)


def _quantizer(quantize: bool):
    return fake_nvfp4 if quantize else _identity


def p_hat(p, quantize: bool = True):
    """fake_nvfp4 of the probabilities in groups of 16 keys (FP32 operands).

    With ``quantize=False`` the quantizer, including the FP32 rounding of its
    operands, is the identity, and the method reduces to textbook attention."""
    return fake_nvfp4(fl32(p), axis=1) if quantize else np.asarray(p, np.float64)


def hats(q, k, v, quantize: bool = True):
    """Q^, K^, V^: fake-quantized along the head dimension."""
    f = _quantizer(quantize)
    return f(q, axis=-1), f(k, axis=-1), f(v, axis=-1)


def _logits(qh_blk, kh, scale, causal, row0):
    s = scale * (qh_blk @ kh.T)
    if causal:
        i = np.arange(row0, row0 + qh_blk.shape[0])[:, None]
        j = np.arange(kh.shape[0])[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def probs(qh, kh, scale, causal, lse=None):
    """Softmax probabilities of one head (Sq, Sk); from ``lse`` if given."""
    s = _logits(qh, kh, scale, causal, 0)
    if lse is None:
        m = np.max(s, axis=1, keepdims=True)
        lse = (m + np.log(np.sum(np.exp(s - m), axis=1, keepdims=True)))[:, 0]
    return np.exp(s - np.asarray(lse, np.float64)[:, None])


def fwd_head(qh, kh, vh, scale, causal, quantize=True, block=ROW_BLOCK):
    """One head of the forward on pre-quantized operands: (O, O', LSE)."""
    Sq = qh.shape[0]
    o = np.empty((Sq, vh.shape[1]))
    o_hp = np.empty_like(o)
    lse = np.empty(Sq)
    for r0 in range(0, Sq, block):
        s = _logits(qh[r0:r0 + block], kh, scale, causal, r0)
        m = np.max(s, axis=1, keepdims=True)
        l = m + np.log(np.sum(np.exp(s - m), axis=1, keepdims=True))
        p = np.exp(s - l)
        o_hp[r0:r0 + block] = p @ vh
        o[r0:r0 + block] = p_hat(p, quantize) @ vh
        lse[r0:r0 + block] = l[:, 0]
    return o, o_hp, lse


def bwd_head(do, qh, kh, vh, o_hp, lse, scale, causal, quantize=True, block=ROW_BLOCK):
    """One head of the backward on pre-quantized operands: (dQ, dK, dV)."""
    delta = np.sum(o_hp * do, axis=1)
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    for r0 in range(0, qh.shape[0], block):
        r1 = r0 + block
        s = _logits(qh[r0:r1], kh, scale, causal, r0)
        p = np.exp(s - lse[r0:r1, None])
        dv += p_hat(p, quantize).T @ do[r0:r1]
        dp = do[r0:r1] @ vh.T
        ds = p * (dp - delta[r0:r1, None])
        dq[r0:r1] = scale * (ds @ kh)
        dk += scale * (ds.T @ qh[r0:r1])
    return dq, dk, dv


def attn_qat_fwd(q, k, v, scale, causal=False, quantize=True):
    """Forward on BHSD float64 arrays: returns (O, O', LSE) in float64."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    if causal and q.shape[2] != k.shape[2]:
        raise ValueError("causal attention needs Sq == Sk")
    qh, kh, vh = hats(q, k, v, quantize)
    B, H, Sq, D = q.shape
    o = np.empty((B, H, Sq, v.shape[3]))
    o_hp = np.empty_like(o)
    lse = np.empty((B, H, Sq))
    for b in range(B):
        for h in range(H):
            o[b, h], o_hp[b, h], lse[b, h] = fwd_head(qh[b, h], kh[b, h], vh[b, h], scale, causal, quantize)
    return o, o_hp, lse


def attn_qat_bwd(do, q, k, v, o_hp, lse, scale, causal=False, quantize=True):
    """Backward on BHSD float64 arrays: returns (dQ, dK, dV) in float64."""
    do, q, k, v, o_hp, lse = (np.asarray(t, np.float64) for t in (do, q, k, v, o_hp, lse))
    if causal and q.shape[2] != k.shape[2]:
        raise ValueError("causal attention needs Sq == Sk")
    qh, kh, vh = hats(q, k, v, quantize)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dq[b, h], dk[b, h], dv[b, h] = bwd_head(do[b, h], qh[b, h], kh[b, h], vh[b, h],
                                                     o_hp[b, h], lse[b, h], scale, causal, quantize)
    return dq, dk, dv


def lse_ohp_head(qh, kh, vh, scale, causal, block=ROW_BLOCK):
    """LSE and O' = P V^ of every row of one head (no quantization work)."""
    Sq = qh.shape[0]
    o_hp = np.empty((Sq, vh.shape[1]))
    lse = np.empty(Sq)
    for r0 in range(0, Sq, block):
        s = _logits(qh[r0:r0 + block], kh, scale, causal, r0)
        m = np.max(s, axis=1, keepdims=True)
        l = m + np.log(np.sum(np.exp(s - m), axis=1, keepdims=True))
        o_hp[r0:r0 + block] = np.exp(s - l) @ vh
        lse[r0:r0 + block] = l[:, 0]
    return o_hp, lse


def fwd_rows(qh, kh, vh, scale, causal, r0, r1, quantize=True):
    """(O, O', LSE) of query rows [r0, r1) of one head (same equations as fwd_head)."""
    s = _logits(qh[r0:r1], kh, scale, causal, r0)
    m = np.max(s, axis=1, keepdims=True)
    l = m + np.log(np.sum(np.exp(s - m), axis=1, keepdims=True))
    p = np.exp(s - l)
    return p_hat(p, quantize) @ vh, p @ vh, l[:, 0]


def dq_rows(do, qh, kh, vh, o_hp, lse, scale, causal, r0, r1):
    """dQ of query rows [r0, r1) of one head: scale * dS K^ over all keys."""
    d = np.sum(o_hp[r0:r1] * do[r0:r1], axis=1)
    p = np.exp(_logits(qh[r0:r1], kh, scale, causal, r0) - lse[r0:r1, None])
    ds = p * (do[r0:r1] @ vh.T - d[:, None])
    return scale * (ds @ kh)


def dkdv_keys(do, qh, kh, vh, o_hp, lse, scale, causal, k0, k1, quantize=True):
    """dK, dV of key rows [k0, k1) of one head, over all query rows.

    k0 must be a multiple of 16 and k1 a multiple of 16 or the key count, so
    that the block holds whole probability groups (groups start at key 0)."""
    if k0 % 16 or (k1 % 16 and k1 != kh.shape[0]):
        raise ValueError("key block must hold whole 16-key groups")
    d = np.sum(o_hp * do, axis=1)
    s = scale * (qh @ kh[k0:k1].T)
    if causal:
        i = np.arange(qh.shape[0])[:, None]
        j = np.arange(k0, k1)[None, :]
        s = np.where(j > i, -np.inf, s)
    p = np.exp(s - lse[:, None])
    dv = p_hat(p, quantize).T @ do
    ds = p * (do @ vh[k0:k1].T - d[:, None])
    dk = scale * (ds.T @ qh)
    return dk, dv


def infer_fwd(q, k, v, scale, causal=False, quantize=True):
    """Inference forward on BHSD float64 arrays: (O, LSE) with O = softmax(scale
    Q^ K^T) V.

    Q and K are NVFP4 (fake_nvfp4 along D, the values an NVFP4-packed tensor
    holds) and V stays BF16, as in the FP4 inference path of the Attn-QAT paper
    summary (Results: block-scaled NVFP4 on QK, BF16 on PV) and the FastVideo
    attn_qat_infer page (fa4_pv_mode "bf16"). No probability quantization."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    if causal and q.shape[2] != k.shape[2]:
        raise ValueError("causal attention needs Sq == Sk")
    f = _quantizer(quantize)
    qh, kh = f(q, axis=-1), f(k, axis=-1)
    B, H, Sq, _ = q.shape
    o = np.empty((B, H, Sq, v.shape[3]))
    lse = np.empty((B, H, Sq))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = lse_ohp_head(qh[b, h], kh[b, h], v[b, h], scale, causal)
    return o, lse


R2_BLOCK_N = 128


R2_P_FORMATS = ("nvfp4", "e5m2", "e4m3")


def _r2_p_hat(p, p_format, quantize):
    """P^ of one key tile's unnormalised P: fake_nvfp4 in 16-key groups, or the
    FP8 cast of the FP8-P variant (both on the FP32 value of P)."""
    if not quantize:
        return np.asarray(p, np.float64)
    if p_format == "nvfp4":
        return p_hat(p, True)
    return fp8_round(fl32(p), p_format)


def r2_rows(qh, kh, vh, scale, causal, r0, r1, block_n=R2_BLOCK_N, quantize=True, p_format="nvfp4"):
    """Recipe R2, the one-pass forward, for query rows [r0, r1) of one head:
    (O, O', LSE).

    This is the variant that the review of the FastVideo pull request "Add
    Attn-QAT training Triton kernels" points at (its FP8-P branch sums the row
    statistic from the unquantized probabilities). Each query row takes the
    key tiles of ``block_n`` keys in order, with an online softmax:

        m_j   = max(m_{j-1}, max_k S_jk)          the exact running max
        P_j   = exp(S_j - m_j)                    unnormalised
        P^_j  = fake_nvfp4(fl32(P_j))             groups of 16 keys of the tile
                (p_format "e5m2" / "e4m3": the FP8 cast fp8(fl32(P_j)) of the
                FP8-P variant, element by element)
        a_j   = exp(m_{j-1} - m_j)
        l_j   = a_j l_{j-1} + rowsum(P_j)         from the unquantized P
        O'_j  = a_j O'_{j-1} + P_j V^_j
        O_j   = a_j O_{j-1} + P^_j V^_j

    with O = O_n / l_n, O' = O'_n / l_n and LSE = m_n + ln l_n. O' and LSE
    equal the standard forward's, so the backward is the same; only O
    differs, because P^ is formed before normalisation."""
    if p_format not in R2_P_FORMATS:
        raise ValueError(f"p_format must be one of {R2_P_FORMATS}")
    s = _logits(qh[r0:r1], kh, scale, causal, r0)
    n, Sk = s.shape[0], s.shape[1]
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, vh.shape[1]))
    acc_hp = np.zeros((n, vh.shape[1]))
    for c0 in range(0, Sk, block_n):
        c1 = min(Sk, c0 + block_n)
        st = s[:, c0:c1]
        m_new = np.maximum(m, np.max(st, axis=1))
        live = np.isfinite(m_new)                      # rows with a key so far
        a = np.where(np.isfinite(m), np.exp(m - np.where(live, m_new, 0.0)), 0.0)
        p = np.where(live[:, None], np.exp(st - np.where(live, m_new, 0.0)[:, None]), 0.0)
        l = a * l + p.sum(axis=1)
        acc = a[:, None] * acc + _r2_p_hat(p, p_format, quantize) @ vh[c0:c1]
        acc_hp = a[:, None] * acc_hp + p @ vh[c0:c1]
        m = m_new
    return acc / l[:, None], acc_hp / l[:, None], m + np.log(l)


def r2_fwd(q, k, v, scale, causal=False, block_n=R2_BLOCK_N, quantize=True, p_format="nvfp4"):
    """Recipe R2 on BHSD float64 arrays: (O, O', LSE) (see r2_rows); Q^, K^,
    V^ are fake_nvfp4 of Q, K, V as in the standard forward; ``p_format``
    picks the probability quantizer ("nvfp4", or "e5m2" / "e4m3" for the
    FP8-P variant)."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    if causal and q.shape[2] != k.shape[2]:
        raise ValueError("causal attention needs Sq == Sk")
    qh, kh, vh = hats(q, k, v, quantize)
    B, H, Sq, _ = q.shape
    o = np.empty((B, H, Sq, v.shape[3]))
    o_hp = np.empty_like(o)
    lse = np.empty((B, H, Sq))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, Sq, ROW_BLOCK):
                r1 = min(Sq, r0 + ROW_BLOCK)
                o[b, h, r0:r1], o_hp[b, h, r0:r1], lse[b, h, r0:r1] = r2_rows(
                    qh[b, h], kh[b, h], vh[b, h], scale, causal, r0, r1, block_n, quantize, p_format)
    return o, o_hp, lse


def nvfp4_codes(x, axis=-1):
    """NVFP4 encoding of x along ``axis``: (E2M1 codes, E4M3 scale codes).

    Codes follow the formats' bit layouts: E2M1 = sign (bit 3) and a 3-bit
    magnitude index into {0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3FN = 4-bit exponent
    (bias 7) and 3-bit mantissa. Values are those of fake_nvfp4; a zero group
    scale gives codes 0 (or 8 for -0)."""
    from .nvfp4 import GROUP, group_scales, quantize_with_scale
    x = np.asarray(x, np.float64)
    xm = np.moveaxis(x, axis, -1)
    n = xm.shape[-1]
    if n % GROUP:
        raise ValueError("the encoded axis must be a multiple of 16")
    s = group_scales(xm, axis=-1)                                   # (..., n/16)
    y = quantize_with_scale(xm, np.repeat(s, GROUP, axis=-1))
    safe = np.where(np.repeat(s, GROUP, axis=-1) == 0, 1.0, np.repeat(s, GROUP, axis=-1))
    mag = np.abs(y) / safe
    idx = np.searchsorted(np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6]), mag)
    codes = (idx | np.where(np.signbit(y), 8, 0)).astype(np.uint8)
    e = np.where(s > 0, np.floor(np.log2(np.where(s > 0, s, 1.0))), 0)
    normal = s >= 2.0 ** -6
    m_norm = np.rint((s / np.exp2(e) - 1) * 8)
    sc = np.where(normal, ((e + 7).astype(np.int64) << 3) | m_norm.astype(np.int64),
                  np.rint(s / 2.0 ** -9).astype(np.int64))
    return np.moveaxis(codes, -1, axis), np.moveaxis(sc.astype(np.uint8), -1, axis)

