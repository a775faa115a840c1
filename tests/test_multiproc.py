"""The multi-rank path of bench.py on CPU: two gloo ranks, each timing its own
replica, must agree on the slowest rank's time and on the whole-job rate."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + 3.0 * rank          # rank 1 is the slow one
        bench.barrier(world)
        m = bench.max_over_ranks(ms, world)
        q.put((rank, m, bench.whole_job_rate(65536, world, m)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [5.0, 5.0]
    assert res[0][2] == res[1][2] == pytest.approx(2 * 65536 / 5e-3)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(1000, 1, 2.0) == pytest.approx(5e5)
