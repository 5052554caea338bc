"""CUDA Attn-QAT at the full workload sizes against the float64 oracle.

c2 (B=1 H=16 S=4096 D=128) is compared in full on every head, over each
whole head and over each 128-row tile of it. c3, c4 and c5
are too large for a whole-tensor float64 oracle, so the first and the last
(b, h) head are checked on sampled outputs the oracle computes one block at
a time: three 64-row query blocks (start, middle, the ragged end) for O, O',
LSE and dQ, and three 64-key blocks (start, middle, end) for dK and dV.

The GPU runs every head in the launch configuration bench.py times. For the
backward, the checked heads get O' and LSE from the oracle (rounded as the
kernels store them); the other heads keep the GPU forward's, so no oracle
input comes from the CUDA path."""
import numpy as np
import pytest

import oracle
from fp4_quantization_aware_gb300 import attnqat, synth
from parity import LSE_TOL, REL_TOL, COS_TOL, assert_tiles, bf16_dev, rel_cos, round_bf16, to_dev

pytestmark = pytest.mark.gpu


def _check(name, got, ref, report):
    rel, cos = rel_cos(got, ref)
    report.append(f"{name}: rel={rel:.2e} cos={cos:.6f} |ref|={np.linalg.norm(ref):.3e}")
    assert rel <= REL_TOL and cos >= COS_TOL, "\n".join(report)
    assert_tiles(name, got, ref)   # every 128-row tile of a whole head (the sampled blocks are 64 rows)


def _blocks(n, size=64, align=16):
    mid = (n // 2) // align * align
    last = max(0, (n - size) // align * align)
    out = []
    for a in (0, mid, last):
        b = min(n, a + size) if a != last else n
        if (a, b) not in out:
            out.append((a, b))
    return out


def _run(name, heads_full=False):
    import torch
    w = synth.workload(name)
    x = synth.inputs(w)
    t = {n: bf16_dev(a) for n, a in x.items()}
    o, o_hp, lse = attnqat.fwd(t["q"], t["k"], t["v"], causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    heads = [(b, h) for b in range(w.B) for h in range(w.H)] if heads_full else [(0, 0), (w.B - 1, w.H - 1)]
    go, gohp, glse = (a.float().cpu().numpy() for a in (o, o_hp, lse))
    ohp_in, lse_in = gohp.copy(), glse.copy()
    ref = {}
    report = []
    for (b, h) in heads:
        qh, kh, vh = oracle.hats(x["q"][b, h].astype(np.float64), x["k"][b, h].astype(np.float64),
                                 x["v"][b, h].astype(np.float64))
        if heads_full:
            ro, rohp, rlse = oracle.fwd_head(qh, kh, vh, w.scale, w.causal)
            _check(f"{name} ({b},{h}) O", go[b, h], ro, report)
            _check(f"{name} ({b},{h}) O'", gohp[b, h], rohp, report)
        else:
            rohp, rlse = oracle.lse_ohp_head(qh, kh, vh, w.scale, w.causal)
            for r0, r1 in _blocks(w.Sq):
                fo, fohp, _ = oracle.fwd_rows(qh, kh, vh, w.scale, w.causal, r0, r1)
                _check(f"{name} ({b},{h}) O[{r0}:{r1}]", go[b, h, r0:r1], fo, report)
                _check(f"{name} ({b},{h}) O'[{r0}:{r1}]", gohp[b, h, r0:r1], fohp, report)
        err = float(np.max(np.abs(glse[b, h] - rlse)))
        report.append(f"{name} ({b},{h}) LSE max abs err {err:.2e}")
        assert err <= LSE_TOL, "\n".join(report)
        ohp_in[b, h] = round_bf16(rohp)
        lse_in[b, h] = rlse.astype(np.float32)
        ref[(b, h)] = (qh, kh, vh)
    dq, dk, dv = attnqat.bwd(t["do"], t["q"], t["k"], t["v"], bf16_dev(ohp_in), to_dev(lse_in.astype(np.float32)),
                             causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    gdq, gdk, gdv = (a.float().cpu().numpy() for a in (dq, dk, dv))
    for (b, h), (qh, kh, vh) in ref.items():
        do = x["do"][b, h].astype(np.float64)
        ohp, ls = ohp_in[b, h].astype(np.float64), lse_in[b, h].astype(np.float64)
        if heads_full:
            rdq, rdk, rdv = oracle.bwd_head(do, qh, kh, vh, ohp, ls, w.scale, w.causal)
            _check(f"{name} ({b},{h}) dQ", gdq[b, h], rdq, report)
            _check(f"{name} ({b},{h}) dK", gdk[b, h], rdk, report)
            _check(f"{name} ({b},{h}) dV", gdv[b, h], rdv, report)
        else:
            for r0, r1 in _blocks(w.Sq):
                rdq = oracle.dq_rows(do, qh, kh, vh, ohp, ls, w.scale, w.causal, r0, r1)
                _check(f"{name} ({b},{h}) dQ[{r0}:{r1}]", gdq[b, h, r0:r1], rdq, report)
            for k0, k1 in _blocks(w.Sk):
                rdk, rdv = oracle.dkdv_keys(do, qh, kh, vh, ohp, ls, w.scale, w.causal, k0, k1)
                _check(f"{name} ({b},{h}) dK[{k0}:{k1}]", gdk[b, h, k0:k1], rdk, report)
                _check(f"{name} ({b},{h}) dV[{k0}:{k1}]", gdv[b, h, k0:k1], rdv, report)
    assert attnqat.device_status() == 0
    print("\n".join(report))


def test_c2_every_head(lib):
    _run("c2", heads_full=True)


@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_full_size_sampled(lib, name):
    _run(name)
