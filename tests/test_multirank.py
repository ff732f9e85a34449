"""The multi-rank bench logic on CPU with two gloo ranks: the barrier, the
max-over-ranks timing reduction and the weak-scaling whole-job value.  No
data-path collective exists: each rank runs an independent problem."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        t = [0.25, 0.5][rank]  # the slower rank decides
        mx = bench.max_over_ranks(dist, t)
        val = bench.whole_job_value(world, 1e12, 10, mx)
        out[rank] = (mx, val)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_the_work():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        # fork: no CUDA context exists in this CPU-only test, and it skips re-importing torch
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="fork")
        res = dict(out)
    assert res[0][0] == pytest.approx(0.5) and res[1][0] == pytest.approx(0.5)
    # 2 ranks x 1 TFLOP x 10 steps in 0.5 s = 40 TFLOP/s
    assert res[0][1] == pytest.approx(40.0) and res[1][1] == pytest.approx(40.0)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(None, 1.5) == 1.5
    assert bench.whole_job_value(1, 2e12, 5, 1.0) == pytest.approx(10.0)
