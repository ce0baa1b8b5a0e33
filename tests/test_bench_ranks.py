"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each an
independent replica, combine into whole-job throughput with the slowest
rank's time (max over ranks) and a barrier."""

import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, lr = bench.dist_env()
    dist = bench.init_dist(w)
    bench.barrier(dist)
    my_seconds = 0.5 + rank                 # rank 1 is the slow one
    worst = bench.reduce_max(dist, my_seconds)
    value = bench.aggregate(100.0, worst, w)
    bench.barrier(dist)
    q.put((r, w, lr, worst, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, lr, worst, value) in enumerate(res):
        assert (r, w, lr) == (rank, world, rank)
        assert worst == 1.5                 # max over ranks
        assert value == 100.0 * 2 / 1.5     # all ranks' units / slowest time


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1) is None
    assert bench.reduce_max(None, 3.0) == 3.0
    assert bench.aggregate(10.0, 2.0, 1) == 5.0
