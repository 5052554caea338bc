"""The bounded-wait abort path of the real attention kernels.

Every barrier wait in the attention kernels gives up after a limit (2 s by
default): the CTA records ATTNQAT_ERR_TIMEOUT in the device error word, lets
its own in-flight TMA copies and MMAs land (teardown waits that keep the 2 s
limit), frees its TMEM and returns, so the context stays usable. Here the
test export attnqat_selftest_set_wait_limit sets the limit to 0, with which a
wait gives up at the first poll that finds its phase incomplete, so every
kernel family's waits run out at once. The test checks that the call
returns, that the device reports the timeout, and that the next call with
the default limit gives
the same outputs as one made before the abort (and, for the QAT forward and
backward, outputs that match the oracle). Nothing here faults or hangs a GPU:
a wait that runs out only ends early."""
import ctypes

import pytest

from fp4_quantization_aware_gb300 import attnqat, synth
from parity import bf16_dev

pytestmark = pytest.mark.gpu

KINDS = ["fwd_d128", "fwd_d64", "bwd_d128", "bwd_d64", "fwd_r2", "infer"]
SHORT_NS = 0
DEFAULT_NS = 2_000_000_000     # ATTNQAT_DEFAULT_WAIT_LIMIT_NS


def _inputs(D, causal):
    import torch
    B, H, S = 1, 2, 512
    t = {n: bf16_dev(synth.random_bf16((B, H, S, D), 300 + i, 2.0 if n == "q" else 1.0))
         for i, n in enumerate(("q", "k", "v", "do"))}
    o, o_hp, lse = attnqat.fwd(t["q"], t["k"], t["v"], causal=causal)
    torch.cuda.synchronize()
    t["o_hp"], t["lse"] = o_hp, lse
    return t


def _call(kind, t, causal):
    if kind.startswith("fwd_d"):
        return list(attnqat.fwd(t["q"], t["k"], t["v"], causal=causal))
    if kind == "fwd_r2":
        return list(attnqat.fwd_r2(t["q"], t["k"], t["v"], causal=causal))
    if kind == "infer":
        return list(attnqat.infer_fwd(t["q"], t["k"], t["v"], causal=causal))
    return list(attnqat.bwd(t["do"], t["q"], t["k"], t["v"], t["o_hp"], t["lse"], causal=causal))


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("kind", KINDS)
def test_short_wait_limit_aborts_and_recovers(lib, kind, causal):
    import torch
    D = 64 if kind.endswith("d64") else 128
    t = _inputs(D, causal)
    ref = [x.clone() for x in _call(kind, t, causal)]
    torch.cuda.synchronize()
    assert attnqat.device_status(clear=True) == 0
    attnqat.check(lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(SHORT_NS)), "set_wait_limit")
    try:
        _call(kind, t, causal)          # enqueued normally; its CTAs give up on the device
        torch.cuda.synchronize()        # ... and return: the stream drains
    finally:
        attnqat.check(lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(DEFAULT_NS)), "set_wait_limit")
    assert attnqat.device_status(clear=True) == 6
    assert attnqat.device_status(clear=True) == 0
    again = _call(kind, t, causal)
    torch.cuda.synchronize()
    assert attnqat.device_status(clear=True) == 0
    for i, (a, b) in enumerate(zip(again, ref)):
        if kind.startswith("bwd") and i == 0:   # dQ: FP32 reduce-adds in any order
            assert (a.float() - b.float()).abs().max().item() <= 1e-2 * b.float().abs().max().item()
        else:
            assert torch.equal(a, b), f"{kind} output {i} differs after the abort"


def test_parity_after_an_abort(lib):
    """After aborted launches, a forward and backward still match the oracle."""
    from test_attn_gpu import run_case
    import torch
    t = _inputs(128, False)
    attnqat.check(lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(SHORT_NS)), "set_wait_limit")
    try:
        _call("fwd_d128", t, False)
        _call("bwd_d128", t, False)
        torch.cuda.synchronize()
    finally:
        attnqat.check(lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(DEFAULT_NS)), "set_wait_limit")
    assert attnqat.device_status(clear=True) == 6
    run_case(1, 2, 384, 384, 128, True, 2.0)


def test_wait_limit_rejects_above_ten_seconds(lib):
    assert lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(10_000_000_001)) == 1
    attnqat.check(lib.attnqat_selftest_set_wait_limit(ctypes.c_uint64(DEFAULT_NS)), "set_wait_limit")
