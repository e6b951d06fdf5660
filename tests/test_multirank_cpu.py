"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, each with its own step
time, must agree on the slowest rank's time and on the whole-job throughput."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [120.0, 150.0][rank]
    slow = bench.max_over_ranks(ms, world)
    q.put((rank, slow, bench.job_value(131072, world, slow)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slow, value in got:
        assert slow == 150.0
        assert abs(value - 2 * 131072 / 0.150) < 1e-6


def test_single_rank_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(1000, 1, 500.0) == 2000.0
