"""Replicas across ranks (the bench's multi-GPU mode) on CPU with gloo:
every rank runs its own workload and the job time is the slowest rank's,
reduced with MAX; the per-rank work does not depend on the world size."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        job_ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        # weak scaling: units processed grow with the world, per-rank work fixed
        flops_rank = 2 * 8 * 4096 * 7168
        value = world * flops_rank / (job_ms * 1e-3) / 1e12
        out[rank] = (job_ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replicas_take_the_slowest_rank(world):
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == out[1][1]
    assert abs(out[0][1] - 2 * 2 * 8 * 4096 * 7168 / 15e-3 / 1e12) < 1e-9


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, None, None) == 3.25
