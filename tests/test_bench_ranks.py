"""Host logic of bench.py's multi-GPU (weak scaling) path, on CPU with gloo.

Two ranks report different times; both must see the slowest one, and the
whole-job throughput is both ranks' work over that time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (t, bench.whole_job_tflops(1e12, world, t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, [3.0, 5.0], out), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        t, v = out[r]
        assert t == 5.0
        assert v == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.whole_job_tflops(2e12, 1, 2.0) == pytest.approx(1000.0)
