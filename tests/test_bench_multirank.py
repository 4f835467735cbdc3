"""The multi-rank host logic of bench.py on CPU with the gloo backend
(world size 2): the job's step time is the slowest rank's, whole-job tokens/s
counts every rank's replica, and the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [120.0, 150.0][rank]
    slowest = bench.max_over_ranks(local_ms, "cpu")
    value = bench.job_throughput(4096, world, slowest, 1000)

    class Args:
        config, steps, warmup = 1, 3, 3
    ref = bench.bench_reference(Args()) if rank == 1 else "skipped"
    out[rank] = (slowest, value, ref)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, value, _ = res[rank]
        assert slowest == 150.0
        assert value == pytest.approx(4096 * 2 / (150.0 / 1e3 / 1000))
    assert res[1][2] is None          # the reference arm does its work on rank 0 only


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, "cpu") == 12.5
    assert bench.job_throughput(100, 1, 1000.0, 10) == pytest.approx(1000.0)
