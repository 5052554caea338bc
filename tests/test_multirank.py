"""The multi-rank bench path on CPU: two gloo ranks agree on the slowest
rank's timings and on the whole-job throughput (weak scaling: every rank runs
its own copy of the workload, with no collective on the data path)."""
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
