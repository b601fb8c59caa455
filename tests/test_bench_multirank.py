"""Multi-rank bench plumbing on CPU (gloo, world size 2): every rank runs its
own copy of the workload (weak scaling, no data-path collective); the step
time reported is the maximum over ranks."""
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


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    r, lr, ws = bench.dist_env()
    bench.dist_init(ws, "gloo")
    bench.barrier(ws)
    t = bench.max_over_ranks(10.0 + rank, ws)
    seed = bench.rank_seed(1000, r)
    seeds = [None] * ws
    dist.all_gather_object(seeds, seed)
    q.put((r, lr, ws, t, seeds))
    dist.destroy_process_group()


def test_two_ranks_max_time_and_distinct_seeds():
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
    for (r, lr, ws, t, seeds) in out:
        assert ws == 2 and lr == r
        assert t == 11.0
        assert len(set(seeds)) == 2


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_seed(7, 0) == 7
