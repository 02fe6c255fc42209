"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks, each timing its
own replica, agree on the slowest rank's time (the whole-job value divides by it)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    slowest = bench.max_over_ranks(0.5 + rank, w)          # rank 1 is the slow one
    steps = 100
    value = w * steps / slowest
    q.put((r, slowest, value))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(ws))
    assert [g[1] for g in got] == [1.5, 1.5]
    assert all(abs(g[2] - 2 * 100 / 1.5) < 1e-9 for g in got)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
