"""Recipe R2 (one-pass forward, each key tile's P fake-quantized before
normalisation) on the GPU against oracle.r2_fwd with 128-key tiles, the
kernel's tile size, with NVFP4 P^ and with the FP8-P variant (E5M2, E4M3). O, O': rel-Frobenius <= 1e-2 and cosine >= 0.999; LSE:
max abs error <= 1e-3. The full-size shapes are checked on sampled row blocks
of their first and last head, in the launch configuration the bench uses."""
import numpy as np
import pytest

import oracle
from fp4_quantization_aware_gb300 import attnqat, synth
from parity import LSE_TOL, REL_TOL, COS_TOL, assert_tiles, bf16_dev, rel_cos

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, Sq, Sk, D, causal, structure)
    (1, 2, 256, 256, 128, False, "iid"),
    (1, 2, 384, 384, 128, True, "iid"),
    (2, 1, 300, 300, 128, True, "outlier"),     # ragged tail, causal, rescaled references
    (1, 2, 200, 520, 128, False, "iid"),        # cross-attention
    (1, 1, 1, 1, 128, False, "iid"),
    (1, 3, 640, 640, 128, False, "peaked"),
    (1, 2, 256, 400, 64, False, "heavy"),
    (1, 2, 320, 320, 64, True, "iid"),
]


def _case(B, H, Sq, Sk, D, causal, structure):
    gain = 4.0 if structure == "peaked" else 1.0
    w = synth.Workload("t", B, H, Sq, Sk, D, causal, 1 / np.sqrt(D),
                       "iid" if structure == "peaked" else structure, gain)
    return w, synth.inputs(w)


def _check(name, got, ref, report):
    rel, cos = rel_cos(got, ref)
    report.append(f"{name}: rel={rel:.2e} cos={cos:.6f}")
    assert rel <= REL_TOL and cos >= COS_TOL, "\n".join(report)
    assert_tiles(name, got, ref)


FP8_CASES = [c for c in CASES if c[2] > 1]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_r2_matches_oracle(lib, case):
    _run_case(case, "nvfp4")


@pytest.mark.parametrize("fmt", ["e5m2", "e4m3"])
@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "x".join(map(str, c)))
def test_r2_fp8_matches_oracle(lib, case, fmt):
    _run_case(case, fmt)


def _run_case(case, fmt):
    import torch
    w, x = _case(*case)
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o, o_hp, lse = attnqat.fwd_r2(q, k, v, causal=w.causal, scale=w.scale, p_format=fmt)
    torch.cuda.synchronize()
    assert attnqat.device_status() == 0
    ro, rohp, rlse = oracle.r2_fwd(x["q"], x["k"], x["v"], w.scale, w.causal, block_n=128, p_format=fmt)
    report = []
    _check("O", o.float().cpu().numpy(), ro, report)
    _check("O'", o_hp.float().cpu().numpy(), rohp, report)
    err = float(np.max(np.abs(lse.cpu().numpy() - rlse)))
    assert err <= LSE_TOL, f"LSE max abs err {err:.3e}"


def test_r2_differs_from_standard_only_in_o(lib):
    """Same O' and LSE as the two-pass forward (the backward's inputs); O
    follows the other recipe (peaked logits keep most probability groups)."""
    import torch
    w, x = _case(1, 2, 640, 640, 128, False, "peaked")
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o2, ohp2, lse2 = attnqat.fwd_r2(q, k, v, scale=w.scale)
    o1, ohp1, lse1 = attnqat.fwd(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    # both round P to BF16, on different scales (normalised vs the running
    # reference), so they differ by two independent roundings
    rel, cos = rel_cos(ohp2.float().cpu().numpy(), ohp1.float().cpu().numpy())
    assert rel <= REL_TOL and cos >= 0.9999
    assert float((lse2 - lse1).abs().max()) <= 1e-4
    ro, _, _ = oracle.r2_fwd(x["q"], x["k"], x["v"], w.scale, False)
    rs, _, _ = oracle.attn_qat_fwd(x["q"], x["k"], x["v"], w.scale, False)
    got = o2.float().cpu().numpy()
    assert rel_cos(got, ro)[0] * 5 < rel_cos(ro, rs)[0]        # nearer its own recipe by far


def test_r2_repeatable(lib):
    import torch
    w, x = _case(1, 4, 1024, 1024, 128, True, "iid")
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    a = attnqat.fwd_r2(q, k, v, causal=True, scale=w.scale)
    b = attnqat.fwd_r2(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert all(torch.equal(s, t) for s, t in zip(a, b))


def _blocks(n, size=64):
    mid = (n // 2) // 16 * 16
    return [(0, size), (mid, mid + size), (n - size, n)]


@pytest.mark.parametrize("name,fmt", [("c2", "nvfp4"), ("c3", "nvfp4"), ("c5", "nvfp4"), ("c2", "e5m2"),
                                      ("c5", "e4m3")])
def test_r2_full_size_sampled(lib, name, fmt):
    import torch
    w = synth.workload(name)
    x = synth.inputs(w)
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o, o_hp, lse = attnqat.fwd_r2(q, k, v, causal=w.causal, scale=w.scale, p_format=fmt)
    torch.cuda.synchronize()
    assert attnqat.device_status() == 0
    go, gohp, glse = (t.float().cpu().numpy() for t in (o, o_hp, lse))
    report = []
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        qh, kh, vh = oracle.hats(x["q"][b, h].astype(np.float64), x["k"][b, h].astype(np.float64),
                                 x["v"][b, h].astype(np.float64))
        for r0, r1 in _blocks(w.Sq):
            ro, rohp, rl = oracle.r2_rows(qh, kh, vh, w.scale, w.causal, r0, r1, p_format=fmt)
            _check(f"{name} ({b},{h}) O[{r0}:{r1}]", go[b, h, r0:r1], ro, report)
            _check(f"{name} ({b},{h}) O'[{r0}:{r1}]", gohp[b, h, r0:r1], rohp, report)
            err = float(np.max(np.abs(glse[b, h, r0:r1] - rl)))
            assert err <= LSE_TOL, f"{name} ({b},{h}) LSE[{r0}:{r1}] {err:.2e}"
    print("\n".join(report))


def test_r2_fp8_is_its_own_recipe(lib):
    """The FP8 variants keep O' and LSE of the NVFP4 one bit for bit (only P^
    changes) and their O differs from it, closer to O' (finer grid)."""
    import torch
    w, x = _case(1, 2, 512, 512, 128, False, "peaked")
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o4, ohp4, lse4 = attnqat.fwd_r2(q, k, v, scale=w.scale)
    for fmt in ("e5m2", "e4m3"):
        o8, ohp8, lse8 = attnqat.fwd_r2(q, k, v, scale=w.scale, p_format=fmt)
        torch.cuda.synchronize()
        assert torch.equal(ohp8, ohp4) and torch.equal(lse8, lse4)
        d8 = (o8.float() - ohp8.float()).norm().item()
        d4 = (o4.float() - ohp4.float()).norm().item()
        assert 0 < d8 < d4, (fmt, d8, d4)


def test_r2_rejects_unknown_p_format(lib):
    import ctypes
    p = attnqat.problem(1, 1, 128, 128, 128)
    x = bf16_dev(np.zeros((1, 1, 128, 128), np.float32))
    ws = attnqat.workspace(lib.attnqat_fwd_workspace_bytes(ctypes.byref(p)), x.device)
    st = lib.attnqat_fwd_r2_p(ctypes.byref(p), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                              x.data_ptr(), 7, ws.data_ptr(), ws.numel(), None)
    assert st == 1
