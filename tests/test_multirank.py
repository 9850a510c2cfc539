"""The N > 1 path of bench.py on CPU: two gloo ranks (spawned processes,
127.0.0.1 rendezvous).  The path shards by replica with no data-path
collective; what crosses ranks is the timing (maximum over ranks) and the
whole-job value, and every rank draws its own inputs."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from block_sparse_attention_tile_gb300 import synthetic


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step time 10 + r ms and e2e 30 - r ms: both ranks must see the maxima
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world)
        # each replica's inputs come from its own seed
        w = bench.WORKLOADS["video_tiny"]
        x = synthetic.normal((4, 8), bench.rank_seed(w["seed"], rank))
        gathered = [torch.empty_like(x) for _ in range(world)]
        dist.all_gather(gathered, x)
        out[rank] = (got, [g.sum().item() for g in gathered])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_seeds():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        got, sums = res[rank]
        assert got == [11.0, 30.0]            # max over ranks of each timing
        assert sums[0] != sums[1]             # replicas draw different inputs
    assert res[0][1] == res[1][1]


def test_job_value_is_weak_scaling_aggregate():
    flops = bench.metric_flops(bench.WORKLOADS["video_dit_bsa"])
    one = bench.job_tflops(flops, 1, 16.0)
    assert bench.job_tflops(flops, 2, 16.0) == pytest.approx(2 * one)
    assert bench.job_tflops(flops, 2, 32.0) == pytest.approx(one)  # the slowest rank sets the time
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
