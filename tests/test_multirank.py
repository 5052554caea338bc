"""The multi-rank paths on CPU with gloo ranks.

Replicas (weak scaling): two ranks agree on the slowest rank's timings and on
the whole-job throughput, every rank running its own copy of the workload.
Data parallel over heads (strong scaling, `bench.py --shard heads`): the
ranks' slices cover every (b, h) head exactly once, contiguously in BHSD, and
slices computed on separate ranks (the oracle standing in for the kernels on
CPU) reassemble to the single-rank result bit for bit. Neither mode has a
collective on the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + rank, 5.0 - rank, 7.0 * (rank + 1)]
        out[rank] = bench.max_over_ranks(local)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [11.0, 5.0, 14.0]


def test_job_throughput_is_weak_scaling_sum():
    # 2 ranks, each 1e12 flop per step, 4 steps, slowest rank 2 ms in total
    assert bench.job_tflops(1e12, 4, 2, 2.0) == pytest.approx(4000.0)
    assert bench.max_over_ranks([1.0, 2.0]) == [1.0, 2.0]      # no process group: unchanged


# ---------------------------------------------------------------- data parallel over B*H heads

@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 40, 64])
def test_head_slices_cover_every_head_once(n):
    for world in range(1, min(n, 8) + 1):
        slices = [bench.head_slice(n, world, r) for r in range(world)]
        assert slices[0][0] == 0 and slices[-1][1] == n
        for (a0, a1), (b0, b1) in zip(slices, slices[1:]):
            assert a1 == b0                                   # contiguous, no gap, no overlap
        sizes = [b - a for a, b in slices]
        assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_shard_heads_are_contiguous_in_bhsd():
    from fp4_quantization_aware_gb300 import synth
    w = synth.workload("c3")                                  # B=2 H=32 S=8192 D=128
    seen = []
    for r in range(3):
        hs = bench.shard_heads(w, 3, r)
        flat = [b * w.H + h for b, h in hs]
        assert flat == list(range(flat[0], flat[0] + len(flat)))
        off = bench.shard_byte_offsets(w, hs)
        assert off["q"] == flat[0] * w.Sq * w.D * 2 and off["k"] == flat[0] * w.Sk * w.D * 2
        assert off["lse"] == flat[0] * w.Sq * 4
        rw = bench.rank_workload(w, hs)
        assert (rw.B, rw.H, rw.Sq, rw.D, rw.causal) == (len(hs), 1, w.Sq, w.D, w.causal)
        seen += flat
    assert seen == list(range(w.B * w.H))
    assert sum(bench.rank_workload(w, bench.shard_heads(w, 3, r)).bwd_flops() for r in range(3)) == w.bwd_flops()
    with pytest.raises(ValueError):
        bench.shard_heads(synth.workload("c1"), 3, 0)         # more ranks than heads


def _shard_rank_main(rank, world, port, out, causal):
    import numpy as np
    import oracle
    from fp4_quantization_aware_gb300 import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.workload("c1", B=2, H=3, Sq=48, Sk=48, causal=causal)
        hs = bench.shard_heads(w, world, rank)
        x = synth.inputs(w, heads=hs)                         # this rank's heads only
        o, o_hp, lse = oracle.attn_qat_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
        dq, dk, dv = oracle.attn_qat_bwd(x["do"], x["q"], x["k"], x["v"], o_hp, lse, w.scale, w.causal)
        parts = [None] * world
        dist.all_gather_object(parts, (hs, [o, o_hp, lse, dq, dk, dv]))
        if rank == 0:
            out["heads"] = [h for p in parts for h in p[0]]
            out["res"] = [np.concatenate([p[1][i] for p in parts]) for i in range(6)]
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal", [False, True])
def test_two_gloo_ranks_reassemble_the_whole_workload(causal):
    """Each rank runs only its slice of heads (generated on its own); put back
    in rank order, the slices give exactly the single-rank result."""
    import numpy as np
    import oracle
    from fp4_quantization_aware_gb300 import synth
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_shard_rank_main, args=(world, port, out, causal), nprocs=world, join=True)
        heads, res = out["heads"], out["res"]
    w = synth.workload("c1", B=2, H=3, Sq=48, Sk=48, causal=causal)
    assert heads == [(b, h) for b in range(w.B) for h in range(w.H)]
    x = synth.inputs(w)
    o, o_hp, lse = oracle.attn_qat_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
    grads = oracle.attn_qat_bwd(x["do"], x["q"], x["k"], x["v"], o_hp, lse, w.scale, w.causal)
    for got, want in zip(res, (o, o_hp, lse) + tuple(grads)):
        want = np.asarray(want).reshape((w.B * w.H, 1) + np.asarray(want).shape[2:])
        assert np.array_equal(got, want)
