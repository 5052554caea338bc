"""CUDA Attn-QAT forward and backward against the float64 oracle (small shapes).

The backward takes the oracle forward's O' and LSE, rounded as the kernels
store them (BF16 and FP32), so no oracle input comes from the CUDA path.
Bounds: relative Frobenius error <= 1e-2 and cosine >= 0.999 on O, O', dQ,
dK, dV; max abs error <= 1e-3 on the natural-log LSE."""
import numpy as np
import pytest

import oracle
from fp4_quantization_aware_gb300 import attnqat, synth
from parity import LSE_TOL, assert_close, bf16_dev, host, round_bf16, to_dev

pytestmark = pytest.mark.gpu

# (B, H, Sq, Sk, D, causal, q_gain)
CASES = [
    (1, 2, 256, 256, 64, False, 1.0),      # the D=64 workload (B1 H2 S256)
    (1, 2, 256, 256, 64, False, 4.0),      # sharpened logits: most P groups survive quantization
    (1, 1, 128, 128, 128, False, 3.0),     # one tile
    (2, 3, 200, 200, 128, True, 3.0),      # causal, ragged tail
    (1, 2, 1, 1, 64, True, 1.0),           # degenerate: one query, one key
    (1, 1, 17, 17, 128, False, 2.0),       # shorter than one key group pair
    (1, 2, 129, 300, 128, False, 2.0),     # cross attention with tails on both axes
    (1, 1, 300, 129, 64, False, 2.0),
    (1, 2, 384, 384, 128, True, 2.0),      # several causal tiles
    (1, 1, 520, 520, 64, True, 3.0),       # tail of 8 rows past four tiles
    (1, 2, 200, 1000, 128, False, 3.0),    # eight key tiles with a ragged last one
]


def make_inputs(B, H, Sq, Sk, D, gain, seed):
    q = synth.random_bf16((B, H, Sq, D), seed, gain)
    k = synth.random_bf16((B, H, Sk, D), seed + 1)
    v = synth.random_bf16((B, H, Sk, D), seed + 2)
    do = synth.random_bf16((B, H, Sq, D), seed + 3)
    return q, k, v, do


def run_case(B, H, Sq, Sk, D, causal, gain, seed=100):
    import torch
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = make_inputs(B, H, Sq, Sk, D, gain, seed)
    tq, tk, tv, tdo = (bf16_dev(a) for a in (q, k, v, do))
    o, o_hp, lse = attnqat.fwd(tq, tk, tv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ro, rohp, rlse = oracle.attn_qat_fwd(q, k, v, scale, causal)
    res = {"O": assert_close("O", host(o), ro), "O'": assert_close("O'", host(o_hp), rohp)}
    lse_err = float(np.max(np.abs(lse.cpu().numpy() - rlse)))
    assert lse_err <= LSE_TOL, f"LSE max abs err {lse_err:.3e}"

    ohp_in = round_bf16(rohp)
    lse_in = rlse.astype(np.float32)
    dq, dk, dv = attnqat.bwd(tdo, tq, tk, tv, bf16_dev(ohp_in), to_dev(lse_in), causal=causal, scale=scale)
    torch.cuda.synchronize()
    rdq, rdk, rdv = oracle.attn_qat_bwd(do, q, k, v, ohp_in, lse_in.astype(np.float64), scale, causal)
    res["dQ"] = assert_close("dQ", host(dq), rdq)
    res["dK"] = assert_close("dK", host(dk), rdk)
    res["dV"] = assert_close("dV", host(dv), rdv)
    assert attnqat.device_status() == 0
    return res


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}D{}{}g{}".format(*c[:5], "c" if c[5] else "", c[6]))
def test_parity_small(lib, case):
    run_case(*case)


def test_outputs_untouched_past_the_tail(lib):
    """Rows past Sq belong to the next head: writes stay inside each head."""
    import torch
    B, H, S, D = 1, 2, 130, 128
    q, k, v, do = make_inputs(B, H, S, S, D, 2.0, 7)
    tq, tk, tv = (bf16_dev(a) for a in (q, k, v))
    o = torch.full((B, H, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_hp = torch.full_like(o, float("nan"))
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    attnqat.fwd(tq, tk, tv, out=(o, o_hp, lse))
    torch.cuda.synchronize()
    assert not torch.isnan(o).any() and not torch.isnan(o_hp).any() and not torch.isnan(lse).any()


def test_repeatable(lib):
    """Two runs on the same inputs agree bit for bit except dQ (atomic order)."""
    import torch
    q, k, v, do = make_inputs(1, 2, 256, 256, 128, 2.0, 9)
    t = [bf16_dev(a) for a in (q, k, v, do)]
    a1 = attnqat.fwd(*t[:3])
    a2 = attnqat.fwd(*t[:3])
    for x, y in zip(a1, a2):
        assert torch.equal(x, y)
    g1 = attnqat.bwd(t[3], *t[:3], a1[1], a1[2])
    g2 = attnqat.bwd(t[3], *t[:3], a1[1], a1[2])
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert (g1[0].float() - g2[0].float()).abs().max().item() <= 1e-2 * g1[0].float().abs().max().item()


def test_bounded_wait_reports_timeout(lib):
    import torch
    assert attnqat.device_status(clear=True) == 0
    attnqat.check(lib.attnqat_selftest_wait_timeout(50_000_000, torch.cuda.current_stream().cuda_stream), "selftest")
    assert attnqat.device_status(clear=True) == 6
    assert attnqat.device_status(clear=True) == 0
    # the context is still usable afterwards
    run_case(1, 1, 128, 128, 64, False, 2.0)


def test_autograd_function_matches_the_c_abi(lib):
    import torch
    q, k, v, do = (bf16_dev(a) for a in make_inputs(1, 2, 200, 200, 128, 2.0, 21))
    q.requires_grad_(), k.requires_grad_(), v.requires_grad_()
    o = attnqat.attention(q, k, v, causal=True)
    o.backward(do)
    o2, o_hp, lse = attnqat.fwd(q.detach(), k.detach(), v.detach(), causal=True)
    dq, dk, dv = attnqat.bwd(do, q.detach(), k.detach(), v.detach(), o_hp, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert torch.equal(k.grad, dk) and torch.equal(v.grad, dv)
    assert (q.grad.float() - dq.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()
