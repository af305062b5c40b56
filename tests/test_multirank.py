"""The benchmark's multi-rank path on the CPU: two gloo ranks (one process each,
as torchrun launches them) agree on the slowest rank's time, pass the barriers,
and the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        bench.barrier(ws)
        t = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))   # rank 1 is the slower one
        value = bench.job_throughput(64, ws, t)
        out[rank] = (ws, r, local, t, value)
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank, (ws, r, local, t, value) in res.items():
        assert (ws, r, local) == (2, rank, rank)
        assert t == 2.5                              # the max over ranks, seen by both
        assert value == pytest.approx(2 * 64 / 2.5e-3)   # whole-job tokens/s: both batches over the slowest


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload, seed, rows, layers, steps, warmup = "decode-1b", 0, None, None, 1, 3
    assert bench.run_reference(Args()) == 0   # returns at once, no work, no output
