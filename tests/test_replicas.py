"""Replicas (multi-GPU is N independent copies of the layer): the host logic
of bench.py's N > 1 run, on CPU with gloo and two processes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took 10 + r ms for the device-timed steps and 30 - r ms end to end
    t = bench.max_over_ranks([10.0 + rank, 30.0 - rank], dist, "cpu")
    out[rank] = t + [bench.job_tokens_per_s(world, 21, 100, t[0])]
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_tokens():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r][:2] == [11.0, 30.0]                 # max over ranks, per entry
        assert res[r][2] == pytest.approx(2 * 21 * 100 / 0.011)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    class A:  # the fields run_reference reads
        steps, warmup, gpus, workload = 1, 0, 2, "decode"
    assert bench.run_reference(A()) == 0   # returns at once, no oracle work, no output


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_tokens_per_s(1, 21, 10, 1.0) == pytest.approx(210000.0)
