"""bench.py's multi-rank host logic on CPU: two gloo ranks (replicas) reduce
their timings to the slowest one, and the whole-job value counts every
rank's bytes over that time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 3.0]
        got = bench.max_over_ranks(mine)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_timing():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert out[0] == out[1] == [2.0, 10.0, 3.0]


def test_whole_job_value_counts_all_ranks():
    import bench
    # 2 ranks x 2 GiB each in 0.5 ms (slowest) -> 8.59 TB/s whole job
    assert bench.whole_job_gbs(2, 2 * 2 ** 30, 0.5) == pytest.approx(2 * 2 * 2 ** 30 / 0.5e-3 / 1e9)
    assert bench.whole_job_gbs(1, 10 ** 9, 1000.0) == pytest.approx(1.0)


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 1.5]) == [3.0, 1.5]
