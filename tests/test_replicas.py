"""The replica (N > 1) host logic of bench.py over gloo on the CPU.

Requests are independent through the whole path, so N GPUs run N independent
replicas: a barrier around the timed region, the slowest rank's time, and the
whole job's throughput = units all ranks processed / that time.  No collective
touches the data path; these tests run the two that the timing uses.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        slowest = bench.max_over_ranks(times[rank], ws)
        out[rank] = (slowest, bench.aggregate_rate(100, slowest, ws))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2, 3])
def test_max_over_ranks_and_rate(ws):
    times = [12.5, 40.0, 7.25][:ws]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(ws, _free_port(), times, out), nprocs=ws, join=True)
        got = dict(out)
    for r in range(ws):
        slowest, rate = got[r]
        assert slowest == max(times)
        assert rate == pytest.approx(ws * 100 / (max(times) * 1e-3))


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.aggregate_rate(10, 20.0, 1) == pytest.approx(500.0)
