"""The multi-rank reduction of bench.py, on two gloo ranks on the CPU.

bench.py under torchrun runs one replica per GPU, times each rank with CUDA events
and reports the slowest rank's time (max over ranks) and the whole-job throughput
(all ranks' bytes over that time).  These tests run the same two functions on two
CPU processes with the gloo backend.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist_env()
        ms = [1.5 + rank, 10.0 - 3 * rank, 7.0]  # per-rank step times (ms)
        got = bench.reduce_max_over_ranks(ms, torch.device("cpu"))
        out[rank] = (ws, r, local, got, bench.whole_job_gbps(ws, 1e9, got[0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_whole_job_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank in range(world):
        ws, r, local, got, gbps = out[rank]
        assert (ws, r, local) == (world, rank, rank)
        assert got == [2.5, 10.0, 7.0]                 # max over ranks, element by element
        assert gbps == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)  # both ranks' bytes over the slowest time


def test_single_process_reduction_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max_over_ranks([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]
    assert bench.whole_job_gbps(1, 164888576, 0.07) == pytest.approx(164888576 / 70e-6 / 1e9)
