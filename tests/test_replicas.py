"""Multi-GPU runs are independent replicas: each rank runs its own group on its
own GPU and no data crosses GPUs. The only cross-rank exchange is the host-side
max of the replicas' times, checked here with world_size 2 on gloo (no GPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        slowest = bench.replica_time(dist, times[rank])
        out[rank] = (slowest, bench.whole_job_rate(world, 1 << 30, slowest))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_time_and_the_sum_of_work():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    times = [2.0, 3.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, rate = out[r]
        assert slowest == 3.0
        assert rate == pytest.approx(2 * (1 << 30) / 3e-3 / 1e9)


def test_single_process_needs_no_group():
    assert bench.replica_time(None, 1.5) == 1.5
    assert bench.whole_job_rate(1, 10 ** 9, 1000.0) == pytest.approx(1.0)
