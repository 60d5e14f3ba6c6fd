"""The benchmark's multi-GPU bookkeeping, exercised with two gloo ranks on the
CPU: replicas share only their timings (max over ranks), never data."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from dense_gemm_07_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank reports different times; the slowest rank sets the pace
        local = [1.0 + rank, 0.5 * (world - rank), 3.0]
        got = replicas.max_over_ranks(local)
        rate = replicas.whole_job_rate(world, 2.0, got[0])
        out.put((rank, got, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in results:
        assert got == [2.0, 1.0, 3.0]           # max over ranks, element-wise
        assert rate == pytest.approx(2 * 2.0 / 2.0)


def test_single_process_is_identity():
    assert replicas.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert replicas.whole_job_rate(4, 10.0, 2.0) == 20.0
    with pytest.raises(ValueError):
        replicas.whole_job_rate(1, 1.0, 0.0)
