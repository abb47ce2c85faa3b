"""The multi-GPU path of bench.py is replicas with no data-path collective:
each rank times its own copy of the step, one all-reduce MAX picks the
slowest rank, and the job's throughput is world x step work over that time.
Checked here with two gloo ranks on CPU; the reference arm does its CPU work
on rank 0 only."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.slowest_rank_ms(ms_by_rank[rank], world, "cpu")
        out[rank] = (ms_max, bench.weak_scaling_tflops(1e12, world, ms_max))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_job_total():
    world, port = 2, _free_port()
    ms_by_rank = [2.0, 5.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, ms_by_rank, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms_max, tflops = res[rank]
        assert ms_max == 5.0                                   # every rank sees the slowest
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)  # world x work / slowest time


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(3.5, 1, "cpu") == 3.5
    assert bench.weak_scaling_tflops(2e12, 1, 4.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"config": "tiny", "warmup": 1, "steps": 1, "gpus": 2, "fwd_only": False})()
    assert bench.run_reference(args) == 0   # returns at once: no oracle work, no output
