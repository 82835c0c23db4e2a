"""bench.py's replica path on two CPU ranks (gloo): the timed value is the max over
ranks and the job throughput counts every rank's work (CPU only)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(100.0 + 50.0 * rank)           # rank 1 is slower
    v = bench.job_throughput(1_000_000_000, 10, world, t)
    out[rank] = (t, v)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    # 2 ranks x 10 steps x 1 GB in the slowest rank's 150 ms
    assert abs(res[0][1] - 2 * 10 / 0.150) < 1e-6


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert abs(bench.job_throughput(4294983680, 100, 1, 61.6621) - 6965.35) < 0.05
