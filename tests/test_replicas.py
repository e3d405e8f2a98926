"""Replicas-only multi-GPU bookkeeping of bench.py, on CPU with the gloo backend: every rank runs its own
drafter replica, the job's time is the slowest rank's, and the job's throughput sums all replicas' tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    import sys
    import torch
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    t = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    out[rank] = t
    out[world + rank] = bench.replica_throughput(world, 15, 10, t)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_throughput(world):
    ctx = mp.get_context("spawn")
    times = [10.0 + 7.5 * r for r in range(world)]
    out = ctx.Array("d", 2 * world)
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    slowest = max(times)
    assert all(out[r] == slowest for r in range(world))
    want = world * 15 * 10 / (slowest / 1e3)
    assert all(abs(out[world + r] - want) < 1e-9 * want for r in range(world))
