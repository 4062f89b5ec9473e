"""The bench's multi-GPU path on CPU: world_size 2 over gloo.  The decode path does not
shard, so N GPUs run N independent replicas; what the ranks share is the barrier, the
slowest rank's time and the whole-job throughput computed from it."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        mine = [0.25, 0.75][rank]                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(mine, torch.device("cpu"))
        value = bench.job_throughput(1_000_000_000, 4, world, slowest)
        results[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        got = dict(results)
    assert got[0] == got[1] == (0.75, 1_000_000_000 * 4 * 2 / 0.75 / 1e9)


def test_job_throughput_counts_every_replica():
    assert bench.job_throughput(10, 3, 4, 2.0) == 10 * 3 * 4 / 2.0 / 1e9
