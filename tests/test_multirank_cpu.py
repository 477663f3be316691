"""The N > 1 host logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own copy of the workload (weak scaling, no data-path
collective); the only collectives are the timing barrier and the max over
ranks. These tests run that logic with world_size 2.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    t = 1.0 + rank          # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, w)
    rate = bench.whole_job_rate(10.0, w, tmax)
    bench.barrier(w)
    q.put((r, w, lr, tmax, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_units():
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
    assert [r[0] for r in res] == [0, 1]
    for r, w, lr, tmax, rate in res:
        assert w == 2 and lr == r
        assert tmax == 2.0                     # max over ranks
        assert rate == pytest.approx(10.0)     # 2 ranks x 10 units / 2 s


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(8.0, 1, 2.0) == 4.0
    assert not dist.is_initialized()
