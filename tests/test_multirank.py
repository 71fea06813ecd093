"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

bench.py under torchrun runs one rank per GPU, each on its own batch of the
workload (weak scaling, no collective on the data path); the only collective
is the max over ranks of the timed duration.  These tests run that logic
with world_size 2 on the gloo backend.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 14.0][rank]
        m = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        seed = bench.rank_seed(0, rank)
        from differential_attention_causal_gb300 import inputs
        x = inputs.make_v1(inputs.V1Shape(1, 4, 1, 8, 0, "fp32"), seed=seed)
        out[rank] = (m, seed, float(x["q"].sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 14.0            # slowest rank sets the time
    assert res[0][1] != res[1][1]                     # each rank its own seed
    assert res[0][2] != res[1][2]                     # ... and so its own batch


def test_job_throughput_is_weak_scaling_aggregate():
    import bench
    one = bench.job_throughput(1e11, 100, 1, 10.0)
    two = bench.job_throughput(1e11, 100, 2, 10.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(1e11 * 100 / 0.01 / 1e12)
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
