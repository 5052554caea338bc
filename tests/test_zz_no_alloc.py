"""attnqat_bwd_noalloc: the backward for callers that cannot allocate device
memory, with its scratch in the library's 32 MiB static device array.

It must give what attnqat_bwd (caller workspace) gives, on two calls in a row
(the second call reuses the array that the first one left behind), and it
must reject problems whose scratch exceeds the array. This file is collected
last so that a run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest

from fp4_quantization_aware_gb300 import attnqat, synth
from parity import assert_close, bf16_dev, host

pytestmark = pytest.mark.gpu


def test_bwd_noalloc_matches_workspace_backward(lib):
    import torch
    B, H, S, D = 1, 2, 384, 128
    p = attnqat.problem(B, H, S, S, D, causal=False)
    assert lib.attnqat_bwd_workspace_bytes(ctypes.byref(p)) <= 32 << 20
    q, k, v, do = (bf16_dev(synth.random_bf16((B, H, S, D), 40 + i, 2.0 if i == 0 else 1.0)) for i in range(4))
    o, o_hp, lse = attnqat.fwd(q, k, v)
    ref = attnqat.bwd(do, q, k, v, o_hp, lse)
    torch.cuda.synchronize()
    ref = [host(t) for t in ref]
    stream = torch.cuda.current_stream().cuda_stream
    outs = [[torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)] for _ in range(2)]
    torch.cuda.synchronize()
    mem0 = torch.cuda.memory_allocated()
    for call in range(2):
        dq, dk, dv = outs[call]
        st = lib.attnqat_bwd_noalloc(ctypes.byref(p), do.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     o_hp.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     stream)
        attnqat.check(st, "attnqat_bwd_noalloc")
        torch.cuda.synchronize()
        # the call allocates nothing: torch's allocator and the device's free
        # memory stay where the first call (which may load the array's module)
        # left them
        if call == 0:
            free0 = torch.cuda.mem_get_info()[0]
        else:
            assert torch.cuda.mem_get_info()[0] == free0
        assert torch.cuda.memory_allocated() == mem0
    for call in range(2):
        for name, got, want in zip(("dQ", "dK", "dV"), outs[call], ref):
            assert_close(f"call {call} {name}", host(got), want)
    assert attnqat.device_status() == 0


def test_bwd_noalloc_rejects_problems_beyond_the_array(lib):
    import torch
    p = attnqat.problem(1, 16, 4096, 4096, 128)
    assert lib.attnqat_bwd_workspace_bytes(ctypes.byref(p)) > 32 << 20
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = lib.attnqat_bwd_noalloc(ctypes.byref(p), *([x.data_ptr()] * 9), torch.cuda.current_stream().cuda_stream)
    assert st == 4
    assert b"32 MiB" in lib.attnqat_last_error_message()
