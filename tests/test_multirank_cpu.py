"""The N > 1 path of bench.py on the CPU: two gloo ranks run independent
replicas (different seeds, no data-path collective); the job time is the
slowest rank's and the throughput counts every rank's work."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [12.0, 30.0][rank]       # rank 1 is the slower replica
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.job_tflops(1e12, world, 10, slowest)
        seed = bench.rank_seed(1003, rank)
        g = torch.Generator().manual_seed(seed)
        sample = torch.randn(4, generator=g)
        gathered = [torch.zeros(4) for _ in range(world)]
        dist.all_gather(gathered, sample)   # test-side check only
        results[rank] = (slowest, value, seed, [t.tolist() for t in gathered])
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_aggregate_throughput():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        r0, r1 = results[0], results[1]
    assert r0[0] == r1[0] == 30.0                       # both see the slowest rank
    assert r0[1] == pytest.approx(2 * 10 * 1e12 / 30e-3 / 1e12)
    assert r0[2] != r1[2]                               # independent replicas
    assert r0[3][0] != r0[3][1]                         # different inputs per rank


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(5.0, 1) == 5.0
    assert bench.job_tflops(2e12, 1, 4, 8.0) == pytest.approx(1000.0)
