"""attnqat_bwd_host (inputs and outputs in pinned host memory, head groups
whose copies overlap the kernels) against the float64 oracle and against
attnqat_bwd on device buffers.

The backward takes the oracle forward's O' and LSE, rounded as the kernels
store them, so no oracle input comes from the CUDA path. Oracle bounds as in
the other parity tests; against attnqat_bwd (the same kernels on the same
heads, only the order of FP32 additions of dQ and of split key tiles'
partial dK, dV differs) the relative Frobenius error is at most 2e-3."""
import ctypes

import numpy as np
import pytest

import oracle
from fp4_quantization_aware_gb300 import attnqat, synth
from parity import assert_close, bf16_dev, host, round_bf16, to_dev

pytestmark = pytest.mark.gpu

# (B, H, Sq, Sk, D, causal, q_gain, chunks)
CASES = [
    (2, 3, 200, 200, 128, True, 3.0, 4),     # 6 heads in 4 groups (2, 2, 2 heads: three groups)
    (1, 4, 256, 300, 64, False, 2.0, 3),     # cross attention with tails, uneven groups
    (1, 5, 384, 384, 128, False, 4.0, 1),    # one group
    (1, 2, 130, 130, 128, False, 2.0, 9),    # more groups than heads: one head per group
]


def pinned(a, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.float32))).to(dtype).pin_memory()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}D{}{}g{}n{}".format(*c[:5], "c" if c[5] else "",
                                                                                       c[6], c[7]))
def test_bwd_host_matches_oracle_and_device_path(lib, case):
    import torch
    B, H, Sq, Sk, D, causal, gain, chunks = case
    scale = 1.0 / np.sqrt(D)
    q = synth.random_bf16((B, H, Sq, D), 300, gain)
    k = synth.random_bf16((B, H, Sk, D), 301)
    v = synth.random_bf16((B, H, Sk, D), 302)
    do = synth.random_bf16((B, H, Sq, D), 303)
    _, rohp, rlse = oracle.attn_qat_fwd(q, k, v, scale, causal)
    ohp_in, lse_in = round_bf16(rohp), rlse.astype(np.float32)

    hin = {"do": pinned(do, torch.bfloat16), "q": pinned(q, torch.bfloat16), "k": pinned(k, torch.bfloat16),
           "v": pinned(v, torch.bfloat16), "o_hp": pinned(ohp_in, torch.bfloat16),
           "lse": torch.from_numpy(lse_in).pin_memory()}
    hout = [torch.full((B, H, n, D), float("nan"), dtype=torch.bfloat16).pin_memory() for n in (Sq, Sk, Sk)]
    p = attnqat.problem(B, H, Sq, Sk, D, causal, scale)
    pp = ctypes.byref(p)
    nbytes = lib.attnqat_bwd_host_workspace_bytes(pp, chunks)
    assert nbytes > 0
    ws = attnqat.workspace(nbytes, "cuda")
    stream = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    for _ in range(2):   # two calls in a row reuse the slots and the library's copy streams
        attnqat.check(lib.attnqat_bwd_host(pp, P(hin["do"]), P(hin["q"]), P(hin["k"]), P(hin["v"]), P(hin["o_hp"]),
                                           P(hin["lse"]), P(hout[0]), P(hout[1]), P(hout[2]), chunks, P(ws),
                                           ws.numel(), stream), "bwd_host")
        torch.cuda.current_stream().synchronize()
        got = [t.float().numpy().astype(np.float64) for t in hout]
        rdq, rdk, rdv = oracle.attn_qat_bwd(do, q, k, v, ohp_in, lse_in.astype(np.float64), scale, causal)
        for name, g, r in (("dQ", got[0], rdq), ("dK", got[1], rdk), ("dV", got[2], rdv)):
            assert_close(name, g, r)
        dq, dk, dv = attnqat.bwd(bf16_dev(do), bf16_dev(q), bf16_dev(k), bf16_dev(v), bf16_dev(ohp_in),
                                 to_dev(lse_in), causal=causal, scale=scale)
        torch.cuda.synchronize()
        for name, g, r in (("dQ", got[0], host(dq)), ("dK", got[1], host(dk)), ("dV", got[2], host(dv))):
            assert_close(name + " vs attnqat_bwd", g, r, rel_tol=2e-3, cos_tol=0.99999)
    assert attnqat.device_status() == 0


def test_bwd_host_rejects_a_small_workspace(lib):
    import torch
    p = attnqat.problem(1, 2, 128, 128, 64)
    pp = ctypes.byref(p)
    need = lib.attnqat_bwd_host_workspace_bytes(pp, 2)
    ws = attnqat.workspace(need, "cuda")
    h = [torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16).pin_memory() for _ in range(8)]
    lse = torch.zeros(1, 2, 128).pin_memory()
    st = lib.attnqat_bwd_host(pp, *[t.data_ptr() for t in h[:5]], lse.data_ptr(), *[t.data_ptr() for t in h[5:8]],
                              2, ws.data_ptr(), need - 256, torch.cuda.current_stream().cuda_stream)
    assert st == 4   # ATTNQAT_ERR_WORKSPACE, before anything is enqueued
