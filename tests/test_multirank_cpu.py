"""The N > 1 host path of bench.py with gloo ranks on the CPU: each rank
times its own independent ring; the job's time is the max over ranks and the
throughput counts every rank's work (weak scaling)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], world)
    tput = bench.whole_job_throughput(1e12, world, ms)
    dist.barrier()
    q.put((rank, ms, tput))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_weak_scaling_throughput(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tput in out:
        assert ms == 20.0                      # every rank sees the slowest
        assert abs(tput - world * 1e12 / 20e-3 / 1e12) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_throughput(2e12, 1, 1000.0) == 2.0
