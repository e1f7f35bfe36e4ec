"""Multi-rank host logic of the benchmark, on CPU with the gloo backend
(world size 2): the timing barrier's max over ranks and the weak-scaling
whole-job rate.  Every rank would run an independent replica of the workload;
there is no data-path collective to test."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_group_and_rate():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    # weak scaling: 2 ranks x 1e9 bytes in the slowest rank's 100 ms -> 20 GB/s
    assert bench.whole_job_rate(1e9, 100.0, 2) == pytest.approx(2e10)
