"""The N>1 bench path on CPU (gloo, world_size 2): each rank draws its own
batch, the job time is the slowest rank's, and whole-job throughput counts
every rank's bytes once.  No GPU and no collective on the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
    m = bench.max_over_ranks(torch, ms, dist, "cpu")
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(1235, rank))
    q.put((rank, m, seeds))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, seeds in out:
        assert m == 15.0                        # max over ranks
        assert len(set(seeds)) == 2             # independent batches per rank
    import bench
    # 2 ranks x 100 steps x 6 MB in 15 ms of the slowest rank
    assert bench.job_throughput(6e6, 100, 2, 15.0) == pytest.approx(6e6 * 200 / 0.015 / 1e9)
