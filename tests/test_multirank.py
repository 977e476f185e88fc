"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each timing its
own (independent) share of the work; the job reports the slowest rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0 + rank, 5.0 - rank]  # rank 1 is slower on the first, faster on the second
        got = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == [3.0, 5.0] and out[1] == [3.0, 5.0]


def test_job_throughput_counts_every_rank():
    f = bench.step_flops()
    assert abs(f - 1.924145348608e12) < 1e3
    one = bench.job_tflops(f, 1, 2.0)
    assert abs(bench.job_tflops(f, 2, 2.0) - 2 * one) < 1e-9
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_reference_arm_runs_on_rank0_only(capsys):
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
