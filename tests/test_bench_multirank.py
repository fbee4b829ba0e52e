"""The benchmark's multi-rank aggregation, on CPU with the gloo backend and two
ranks: the job time is the slowest rank's and the value counts every rank's
work (weak scaling, one independent replica per rank)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = [10.0, 25.0][rank]          # rank 1 is slower
        ms_max, value = bench.aggregate_ranks(torch, dist, ms, 2e12, 4, "cpu")
        out[rank] = (ms_max, value)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    port = _free_port()
    # spawn, not fork: earlier tests in this process may have started threads
    # (the oracle's OpenMP pool), and a fork of a threaded process can hang.
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ms_max, value = res[rank]
        assert ms_max == 25.0
        # 2 ranks x 4 steps x 2 TFLOP in 25 ms
        assert value == pytest.approx(2 * 4 * 2e12 / 0.025 / 1e12)


def test_aggregate_single_rank():
    import bench
    ms_max, value = bench.aggregate_ranks(torch, None, 8.0, 1e12, 2, "cpu")
    assert ms_max == 8.0 and value == pytest.approx(2 * 1e12 / 0.008 / 1e12)
