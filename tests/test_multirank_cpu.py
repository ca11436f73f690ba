"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): the
slowest rank's time sets the job time, throughput sums the ranks' work, and
every (rank, replica) draws its own batch."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    t = bench.reduce_max(1.0 + rank, w)            # rank 1 is the slow one
    gbs = bench.aggregate(100e6, 10, t, w)         # 100 MB per step per rank, 10 steps
    seeds = [bench.rank_seed(7, r, k) for k in range(3)]
    allseeds = [None] * w
    dist.all_gather_object(allseeds, seeds)
    q.put((r, w, lr, t, gbs, allseeds))
    dist.destroy_process_group()


def test_two_ranks_reduce_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, lr, t, gbs, allseeds) in enumerate(res):
        assert (rank, world, lr) == (r, 2, r)
        assert t == 2.0                             # max over ranks
        assert abs(gbs - 100e6 * 10 * 2 / 2.0 / 1e9) < 1e-9
        flat = [s for rs in allseeds for s in rs]
        assert len(set(flat)) == len(flat)          # no two replicas share data


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate(1e9, 2, 1.0, 1) == 2.0
