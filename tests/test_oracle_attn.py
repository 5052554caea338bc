"""Pins of the oracle's Attn-QAT forward and backward.

Each check uses something other than the oracle's own formulas:

* with the quantizer switched to identity the method is textbook attention, so
  the oracle must match torch's scaled_dot_product_attention and its autograd
  backward in float64;
* dQ and dK are the gradients of the STE surrogate <dO, softmax(scale Q^K^T) V^>
  with respect to Q^ and K^: central finite differences;
* <dO, fake(P) V^> is linear in V^, so dV = fake(P)^T dO is pinned exactly by a
  perturbation of V^;
* the FlashAttention identity rowsum(P * dO V^T) = rowsum(O' * dO) holds exactly
  for the auxiliary output O' (Attn-QAT paper summary, Fix 1);
* the first causal row attends only key 0, so P^ of that row is the one-hot
  group [1.03125, 0, ...] and O_0 = 1.03125 V^_0, O'_0 = V^_0 (closed form);
* a pure-Python brute force on a tiny ragged case (key groups of 16 + 4) with
  an enumeration quantizer.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn, nvfp4
from fp4_quantization_aware_gb300 import synth

from test_oracle_nvfp4 import brute_group


def _inputs(B, H, Sq, Sk, D, seed, gain=1.0):
    rng = np.random.default_rng(seed)
    f = lambda *s: synth.bf16_round(rng.standard_normal(s, dtype=np.float32)).astype(np.float64)
    q = f(B, H, Sq, D) * gain
    return q, f(B, H, Sk, D), f(B, H, Sk, D), f(B, H, Sq, D)


@pytest.mark.parametrize("Sq,Sk,causal", [(40, 40, False), (37, 37, True), (24, 53, False)])
def test_identity_quantizer_matches_sdpa(Sq, Sk, causal):
    q, k, v, do = _inputs(2, 3, Sq, Sk, 16, 11)
    scale = 0.3
    o, o_hp, lse = attn.attn_qat_fwd(q, k, v, scale, causal, quantize=False)
    tq, tk, tv = (torch.tensor(t, requires_grad=True) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    ref.backward(torch.tensor(do))
    np.testing.assert_allclose(o, ref.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o_hp, ref.detach().numpy(), rtol=1e-12, atol=1e-12)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        s = np.where(np.triu(np.ones((Sq, Sk), bool), 1), -np.inf, s)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.tensor(s), -1).numpy(), rtol=1e-13)
    dq, dk, dv = attn.attn_qat_bwd(do, q, k, v, o_hp, lse, scale, causal, quantize=False)
    for got, want in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-11)


def _surrogate(qh, kh, vh, do, scale, causal):
    p = attn.probs(qh, kh, scale, causal)
    return float(np.sum(do * (p @ vh)))


@pytest.mark.parametrize("causal", [False, True])
def test_dq_dk_finite_differences(causal):
    q, k, v, do = _inputs(1, 1, 33, 33, 16, 12)
    scale = 1 / 4
    qh, kh, vh = (nvfp4.fake_nvfp4(t[0, 0]) for t in (q, k, v))
    do = do[0, 0]
    o, o_hp, lse = attn.fwd_head(qh, kh, vh, scale, causal)
    dq, dk, dv = attn.bwd_head(do, qh, kh, vh, o_hp, lse, scale, causal)
    rng = np.random.default_rng(0)
    h = 1e-5
    for target, grad in ((qh, dq), (kh, dk)):
        for _ in range(25):
            i, j = rng.integers(target.shape[0]), rng.integers(target.shape[1])
            old = target[i, j]
            target[i, j] = old + h
            lp = _surrogate(qh, kh, vh, do, scale, causal)
            target[i, j] = old - h
            lm = _surrogate(qh, kh, vh, do, scale, causal)
            target[i, j] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[i, j]) <= 1e-7 * (1 + abs(fd)), (i, j, fd, grad[i, j])


@pytest.mark.parametrize("causal", [False, True])
def test_dv_is_exact_gradient_in_vhat(causal):
    q, k, v, do = _inputs(1, 1, 48, 48, 16, 13, gain=3.0)
    scale = 1 / 4
    qh, kh, vh = (nvfp4.fake_nvfp4(t[0, 0]) for t in (q, k, v))
    do = do[0, 0]
    o, o_hp, lse = attn.fwd_head(qh, kh, vh, scale, causal)
    _, _, dv = attn.bwd_head(do, qh, kh, vh, o_hp, lse, scale, causal)
    assert np.abs(o).max() > 0.1                  # P^ is not all zero here
    e = np.random.default_rng(1).standard_normal(vh.shape)
    o2, _, _ = attn.fwd_head(qh, kh, vh + e, scale, causal)
    lhs = float(np.sum(do * (o2 - o)))
    rhs = float(np.sum(dv * e))
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(rhs))


@pytest.mark.parametrize("causal", [False, True])
def test_flash_identity_with_auxiliary_output(causal):
    q, k, v, do = _inputs(1, 1, 64, 64, 32, 14)
    scale = 1 / math.sqrt(32)
    qh, kh, vh = (nvfp4.fake_nvfp4(t[0, 0]) for t in (q, k, v))
    do = do[0, 0]
    o, o_hp, lse = attn.fwd_head(qh, kh, vh, scale, causal)
    p = attn.probs(qh, kh, scale, causal)
    lhs = np.sum(p * (do @ vh.T), axis=1)
    np.testing.assert_allclose(lhs, np.sum(o_hp * do, axis=1), rtol=1e-12, atol=1e-12)
    # the identity is broken by the quantized output, which is why O' exists
    assert np.max(np.abs(lhs - np.sum(o * do, axis=1))) > 1e-3


def test_causal_first_row_closed_form():
    q, k, v, _ = _inputs(1, 2, 20, 20, 16, 15)
    scale = 0.25
    o, o_hp, lse = attn.attn_qat_fwd(q, k, v, scale, causal=True)
    qh, kh, vh = attn.hats(q, k, v)
    np.testing.assert_array_equal(o[:, :, 0], 1.03125 * vh[:, :, 0])
    np.testing.assert_allclose(o_hp[:, :, 0], vh[:, :, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], scale * np.sum(qh[:, :, 0] * kh[:, :, 0], -1), rtol=1e-14)


def _brute_attention(q, k, v, do, scale, causal):
    """Scalar pure-Python Attn-QAT on one head, with the enumeration quantizer."""
    Sq, D = len(q), len(q[0])
    Sk = len(k)
    qh = [list(brute_group(row[g:g + 16])) for row in q for g in range(0, D, 16)]
    qh = [sum(qh[r * (D // 16):(r + 1) * (D // 16)], []) for r in range(Sq)]
    kh = [sum((list(brute_group(row[g:g + 16])) for g in range(0, D, 16)), []) for row in k]
    vh = [sum((list(brute_group(row[g:g + 16])) for g in range(0, D, 16)), []) for row in v]
    P, Ph, lse = [], [], []
    for i in range(Sq):
        s = [scale * sum(qh[i][d] * kh[j][d] for d in range(D)) if not (causal and j > i) else -math.inf
             for j in range(Sk)]
        m = max(s)
        l = m + math.log(sum(math.exp(x - m) for x in s))
        p = [math.exp(x - l) for x in s]
        p32 = [float(np.float32(x)) for x in p]
        ph = []
        for g in range(0, Sk, 16):
            seg = p32[g:g + 16]
            ph += list(brute_group(seg + [0.0] * (16 - len(seg))))[:len(seg)]
        P.append(p), Ph.append(ph), lse.append(l)
    O = [[sum(Ph[i][j] * vh[j][d] for j in range(Sk)) for d in range(D)] for i in range(Sq)]
    Ohp = [[sum(P[i][j] * vh[j][d] for j in range(Sk)) for d in range(D)] for i in range(Sq)]
    delta = [sum(Ohp[i][d] * do[i][d] for d in range(D)) for i in range(Sq)]
    dP = [[sum(do[i][d] * vh[j][d] for d in range(D)) for j in range(Sk)] for i in range(Sq)]
    dS = [[P[i][j] * (dP[i][j] - delta[i]) for j in range(Sk)] for i in range(Sq)]
    dQ = [[scale * sum(dS[i][j] * kh[j][d] for j in range(Sk)) for d in range(D)] for i in range(Sq)]
    dK = [[scale * sum(dS[i][j] * qh[i][d] for i in range(Sq)) for d in range(D)] for j in range(Sk)]
    dV = [[sum(Ph[i][j] * do[i][d] for i in range(Sq)) for d in range(D)] for j in range(Sk)]
    return [np.array(t) for t in (O, Ohp, lse, dQ, dK, dV)]


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_ragged_brute_force(causal):
    q, k, v, do = _inputs(1, 1, 20, 20, 16, 16, gain=3.0)
    scale = 0.5
    o, o_hp, lse = attn.attn_qat_fwd(q, k, v, scale, causal)
    dq, dk, dv = attn.attn_qat_bwd(do, q, k, v, o_hp, lse, scale, causal)
    want = _brute_attention(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), do[0, 0].tolist(), scale, causal)
    for got, ref in zip((o, o_hp, lse, dq, dk, dv), want):
        np.testing.assert_allclose(got[0, 0], ref, rtol=1e-10, atol=1e-12)
    assert np.count_nonzero(o) > 0


def test_rejects_causal_cross_attention():
    q, k, v, _ = _inputs(1, 1, 8, 12, 16, 17)
    with pytest.raises(ValueError):
        attn.attn_qat_fwd(q, k, v, 0.25, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_row_and_key_blocks_agree_with_whole_head(causal):
    """The sampled-block helpers used at full size equal slices of the whole-head oracle."""
    q, k, v, do = _inputs(1, 1, 70, 70, 16, 18, gain=3.0)
    scale = 0.4
    qh, kh, vh = (nvfp4.fake_nvfp4(t[0, 0]) for t in (q, k, v))
    do = do[0, 0]
    o, o_hp, lse = attn.fwd_head(qh, kh, vh, scale, causal)
    dq, dk, dv = attn.bwd_head(do, qh, kh, vh, o_hp, lse, scale, causal)
    o2, ohp2 = attn.lse_ohp_head(qh, kh, vh, scale, causal)
    np.testing.assert_allclose(o2, o_hp, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(ohp2, lse, rtol=1e-13)
    for r0, r1 in ((0, 5), (30, 47), (60, 70)):
        fo, fohp, flse = attn.fwd_rows(qh, kh, vh, scale, causal, r0, r1)
        np.testing.assert_allclose(fo, o[r0:r1], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(fohp, o_hp[r0:r1], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(flse, lse[r0:r1], rtol=1e-13)
        np.testing.assert_allclose(attn.dq_rows(do, qh, kh, vh, o_hp, lse, scale, causal, r0, r1), dq[r0:r1],
                                   rtol=1e-10, atol=1e-13)
    for k0, k1 in ((0, 16), (32, 64), (64, 70)):
        bk, bv = attn.dkdv_keys(do, qh, kh, vh, o_hp, lse, scale, causal, k0, k1)
        np.testing.assert_allclose(bk, dk[k0:k1], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(bv, dv[k0:k1], rtol=1e-10, atol=1e-13)
    with pytest.raises(ValueError):
        attn.dkdv_keys(do, qh, kh, vh, o_hp, lse, scale, causal, 8, 24)


@pytest.mark.parametrize("causal", [False, True])
def test_infer_fwd_identity_matches_sdpa(causal):
    q, k, v, _ = _inputs(1, 2, 45, 45, 16, 19)
    o, lse = attn.infer_fwd(q, k, v, 0.3, causal, quantize=False)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v),
                                                           is_causal=causal, scale=0.3)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_infer_fwd_is_the_auxiliary_output_with_bf16_v():
    """softmax(scale Q^K^T) V with V unquantized equals O' of the pinned
    training forward run on the same Q^, K^ and an unquantized V."""
    q, k, v, _ = _inputs(2, 2, 40, 40, 32, 20, gain=2.0)
    o, lse = attn.infer_fwd(q, k, v, 0.25, causal=True)
    qh, kh, _ = attn.hats(q, k, v)
    for b in range(2):
        for h in range(2):
            _, o_hp, l2 = attn.fwd_head(qh[b, h], kh[b, h], v[b, h], 0.25, True)
            np.testing.assert_allclose(o[b, h], o_hp, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(lse[b, h], l2, rtol=1e-13)


def test_nvfp4_codes_decode_to_fake_quantized_values():
    from test_oracle_nvfp4 import E2, E4
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal((64, 32)) * 3, rng.standard_normal((8, 32)) * 1e-4,
                        rng.standard_normal((8, 32)) * 5000]).astype(np.float32).astype(np.float64)
    x[0, 5] = -0.0
    codes, sc = attn.nvfp4_codes(x)
    assert codes.shape == x.shape and sc.shape == (x.shape[0], x.shape[1] // 16)
    assert codes.max() <= 15 and sc.max() <= 126
    mag = E2[codes & 7] * np.repeat(E4[sc], 16, axis=1)
    dec = np.where(codes & 8, -mag, mag)
    np.testing.assert_array_equal(dec.view(np.int64), nvfp4.fake_nvfp4(x).view(np.int64))


# ------------------------------------------------------------------ recipe R2
def _golden_rows(name):
    import math
    path = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = []
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        tag, bn, logits, c_r2, c_std = (f.strip() for f in line.split("|"))

        def vals(txt):
            out = []
            for tok in txt.split(","):
                tok = tok.strip()
                rep = 1
                if "*" in tok:
                    tok, rep = tok.split("*")
                    rep = int(rep)
                out += [float(eval(tok, {"__builtins__": {}}, {"ln2": math.log(2.0)}))] * rep
            return np.array(out)
        rows.append((tag, int(bn), vals(logits), vals(c_r2), vals(c_std)))
    return rows


@pytest.mark.parametrize("case", _golden_rows("r2_worked.txt"), ids=lambda c: c[0])
def test_r2_worked_examples(case):
    """Hand-derived R2 outputs (tests/golden/r2_worked.txt): one query row whose
    logits are given directly (Q^ = e_0, K^_j = S_j e_0, scale 1), V^ = identity."""
    _, bn, logits, c_r2, c_std = case
    Sk = len(logits)
    qh = np.zeros((1, 16)); qh[0, 0] = 1.0
    kh = np.zeros((Sk, 16)); kh[:, 0] = logits
    vh = np.eye(Sk)
    o, o_hp, lse = attn.r2_rows(qh, kh, vh, 1.0, False, 0, 1, block_n=bn)
    np.testing.assert_allclose(o[0], c_r2, rtol=1e-12, atol=1e-12)
    o_std, _, _ = attn.fwd_rows(qh, kh, vh, 1.0, False, 0, 1)
    np.testing.assert_allclose(o_std[0], c_std, rtol=1e-12, atol=1e-12)
    p = np.exp(logits - logits.max())
    np.testing.assert_allclose(o_hp[0], p / p.sum(), rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_r2_identity_matches_sdpa(causal):
    q, k, v, _ = _inputs(1, 2, 45, 45, 16, 31)
    o, o_hp, lse = attn.r2_fwd(q, k, v, 0.3, causal, block_n=16, quantize=False)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v),
                                                           is_causal=causal, scale=0.3).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o_hp, ref, rtol=1e-12, atol=1e-12)


def test_r2_auxiliary_outputs_are_the_standard_ones():
    """The online rescaling leaves O' = P V^ and the LSE exactly those of the
    standard forward (the backward's inputs), whatever the tile size."""
    q, k, v, _ = _inputs(1, 2, 70, 70, 32, 32, gain=2.0)
    o_s, ohp_s, lse_s = attn.attn_qat_fwd(q, k, v, 0.2, True)
    for bn in (16, 32, 128):
        o, o_hp, lse = attn.r2_fwd(q, k, v, 0.2, True, block_n=bn)
        np.testing.assert_allclose(o_hp, ohp_s, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse, lse_s, rtol=1e-13)
        assert np.linalg.norm(o - o_s) > 1e-3 * np.linalg.norm(o_s)   # O is a different recipe


def _brute_r2(q, k, v, scale, causal, bn):
    """Scalar pure-Python recipe R2 on one head with the enumeration quantizer."""
    Sq, D, Sk = len(q), len(q[0]), len(k)
    quant = lambda row: sum((list(brute_group(row[g:g + 16])) for g in range(0, len(row), 16)), [])
    qh, kh, vh = [quant(r) for r in q], [quant(r) for r in k], [quant(r) for r in v]
    O, Ohp, L = [], [], []
    for i in range(Sq):
        m, l = -math.inf, 0.0
        acc, acc_hp = [0.0] * D, [0.0] * D
        for c0 in range(0, Sk, bn):
            keys = range(c0, min(Sk, c0 + bn))
            s = [scale * sum(qh[i][d] * kh[j][d] for d in range(D)) if not (causal and j > i) else -math.inf
                 for j in keys]
            m_new = max([m] + s)
            a = math.exp(m - m_new) if m > -math.inf else 0.0
            p = [math.exp(x - m_new) if x > -math.inf else 0.0 for x in s]
            p32 = [float(np.float32(x)) for x in p]
            ph = []
            for g in range(0, len(p32), 16):
                seg = p32[g:g + 16]
                ph += list(brute_group(seg + [0.0] * (16 - len(seg))))[:len(seg)]
            l = a * l + sum(p)
            acc = [a * acc[d] + sum(ph[t] * vh[j][d] for t, j in enumerate(keys)) for d in range(D)]
            acc_hp = [a * acc_hp[d] + sum(p[t] * vh[j][d] for t, j in enumerate(keys)) for d in range(D)]
            m = m_new
        O.append([x / l for x in acc]), Ohp.append([x / l for x in acc_hp]), L.append(m + math.log(l))
    return np.array(O), np.array(Ohp), np.array(L)


@pytest.mark.parametrize("Sq,causal", [(6, False), (40, True)])
def test_r2_matches_brute_force(Sq, causal):
    """Three key tiles of 16 (the last ragged), causal diagonals included."""
    q, k, v, _ = _inputs(1, 1, Sq, 40, 16, 33, gain=3.0)
    bo, bohp, bl = _brute_r2(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.25, causal, 16)
    o, o_hp, lse = attn.r2_fwd(q, k, v, 0.25, causal, block_n=16)
    np.testing.assert_allclose(o[0, 0], bo, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(o_hp[0, 0], bohp, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], bl, rtol=1e-12)


# ------------------------------------------------------------------ recipe R2, FP8-P variant
def _fp8_golden_rows():
    path = os.path.join(os.path.dirname(__file__), "golden", "r2_fp8_worked.txt")
    rows = []
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        tag, fmt, bn, logits, c = (f.strip() for f in line.split("|"))

        def vals(txt):
            out = []
            for tok in txt.split(","):
                tok = tok.strip()
                rep = 1
                if "*" in tok and tok.rsplit("*", 1)[1].isdigit():
                    tok, rep = tok.rsplit("*", 1)
                    rep = int(rep)
                out += [float(eval(tok, {"__builtins__": {}}, {"ln": math.log}))] * rep
            return np.array(out)
        rows.append((tag, fmt, int(bn), vals(logits), vals(c)))
    return rows


@pytest.mark.parametrize("case", _fp8_golden_rows(), ids=lambda c: c[0])
def test_r2_fp8_worked_examples(case):
    """Hand-derived FP8-P outputs (tests/golden/r2_fp8_worked.txt): one query
    row with given logits (Q^ = e_0, K^_j = S_j e_0, scale 1), V^ = identity."""
    _, fmt, bn, logits, c = case
    Sk = len(logits)
    qh = np.zeros((1, 16)); qh[0, 0] = 1.0
    kh = np.zeros((Sk, 16)); kh[:, 0] = logits
    vh = np.eye(Sk)
    o, o_hp, lse = attn.r2_rows(qh, kh, vh, 1.0, False, 0, 1, block_n=bn, p_format=fmt)
    np.testing.assert_allclose(o[0], c, rtol=1e-12, atol=1e-12)
    p = np.exp(logits - logits.max())
    np.testing.assert_allclose(o_hp[0], p / p.sum(), rtol=1e-12)


def _brute_fp8(x, fmt):
    """Nearest FP8 value by enumeration of the format's codes, ties to even."""
    from test_oracle_fp8 import brute
    return float(brute([x], fmt)[0])


def _brute_r2_fp8(q, k, v, scale, causal, bn, fmt):
    """Scalar pure-Python FP8-P recipe R2 on one head (enumeration quantizers)."""
    Sq, D, Sk = len(q), len(q[0]), len(k)
    quant = lambda row: sum((list(brute_group(row[g:g + 16])) for g in range(0, len(row), 16)), [])
    qh, kh, vh = [quant(r) for r in q], [quant(r) for r in k], [quant(r) for r in v]
    O, Ohp, L = [], [], []
    for i in range(Sq):
        m, l = -math.inf, 0.0
        acc, acc_hp = [0.0] * D, [0.0] * D
        for c0 in range(0, Sk, bn):
            keys = range(c0, min(Sk, c0 + bn))
            s = [scale * sum(qh[i][d] * kh[j][d] for d in range(D)) if not (causal and j > i) else -math.inf
                 for j in keys]
            m_new = max([m] + s)
            a = math.exp(m - m_new) if m > -math.inf else 0.0
            p = [math.exp(x - m_new) if x > -math.inf else 0.0 for x in s]
            ph = [_brute_fp8(float(np.float32(x)), fmt) for x in p]
            l = a * l + sum(p)
            acc = [a * acc[d] + sum(ph[t] * vh[j][d] for t, j in enumerate(keys)) for d in range(D)]
            acc_hp = [a * acc_hp[d] + sum(p[t] * vh[j][d] for t, j in enumerate(keys)) for d in range(D)]
            m = m_new
        O.append([x / l for x in acc]), Ohp.append([x / l for x in acc_hp]), L.append(m + math.log(l))
    return np.array(O), np.array(Ohp), np.array(L)


@pytest.mark.parametrize("fmt", ["e5m2", "e4m3"])
@pytest.mark.parametrize("Sq,causal", [(5, False), (36, True)])
def test_r2_fp8_matches_brute_force(Sq, causal, fmt):
    q, k, v, _ = _inputs(1, 1, Sq, 36, 16, 34, gain=3.0)
    bo, bohp, bl = _brute_r2_fp8(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(), 0.25, causal, 16, fmt)
    o, o_hp, lse = attn.r2_fwd(q, k, v, 0.25, causal, block_n=16, p_format=fmt)
    np.testing.assert_allclose(o[0, 0], bo, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(o_hp[0, 0], bohp, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], bl, rtol=1e-12)


@pytest.mark.parametrize("fmt", ["e5m2", "e4m3"])
def test_r2_fp8_identity_and_auxiliary_outputs(fmt):
    """With identity quantizers every P format is textbook attention; O' and
    LSE do not depend on the P format; O does, and the FP8 O lies closer to
    O' than the NVFP4 one (finer probability grid)."""
    q, k, v, _ = _inputs(1, 2, 45, 45, 16, 35)
    o, _, _ = attn.r2_fwd(q, k, v, 0.3, True, block_n=16, quantize=False, p_format=fmt)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v),
                                                           is_causal=True, scale=0.3).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    q, k, v, _ = _inputs(1, 2, 70, 70, 32, 36, gain=2.0)
    o4, ohp4, lse4 = attn.r2_fwd(q, k, v, 0.2, False, block_n=32)
    o8, ohp8, lse8 = attn.r2_fwd(q, k, v, 0.2, False, block_n=32, p_format=fmt)
    np.testing.assert_allclose(ohp8, ohp4, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse8, lse4, rtol=1e-14)
    assert np.linalg.norm(o8 - ohp8) < np.linalg.norm(o4 - ohp4)
