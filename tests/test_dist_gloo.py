"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing
its own replica of the workload, agree on the slowest rank's time and the
whole-job microseconds per call."""
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
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    r, w, _ = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    elapsed = 1.0 + rank                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(elapsed)
    out[rank] = (slowest, bench.whole_job_us_per_call(slowest, 100, w))
    bench.barrier()
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_max_and_whole_job_rate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1]
    slowest, us = out[0]
    assert slowest == 2.0
    # 2 ranks x 100 calls in the slowest rank's 2 s
    assert us == pytest.approx(2.0e6 / 200)


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_us_per_call(0.5, 1000, 1) == pytest.approx(500.0)
