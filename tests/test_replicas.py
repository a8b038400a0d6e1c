"""Weak-scaling bookkeeping of bench.py's N-GPU mode, on CPU with two gloo ranks:
every rank reports the slowest rank's time, and the job throughput counts the work of
all ranks over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_expert_gb300.replicas import job_throughput, max_over_ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower replica
    slowest = max_over_ranks(local_ms)
    out[rank] = (slowest, job_throughput(100.0, world, slowest * 1e-3))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, thr = out[0]
    assert slowest == pytest.approx(15.0)
    assert thr == pytest.approx(100.0 * 2 / 0.015)


def test_single_process_is_its_own_slowest():
    assert max_over_ranks(3.5) == 3.5
    assert job_throughput(10.0, 1, 2.0) == 5.0
