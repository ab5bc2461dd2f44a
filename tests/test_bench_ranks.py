"""The benchmark's multi-rank host logic on CPU with the gloo backend (world size 2).

Ranks are independent replicas: each draws its own batch, the job time is the
slowest rank's, and throughput is the sum over ranks.  No GPU is involved.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from flash_exact_attention_gb300.synth import make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports timings (r + 1, 10 - r): the element-wise max is taken
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist, "cpu")
        x = make_inputs(1, 2, 2, 16, 64, seed=bench.rank_seed(0, rank))
        out[rank] = (got, x["q"].tobytes())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_draw_their_own_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == [2.0, 10.0] and res[1][0] == [2.0, 10.0]
    assert res[0][1] != res[1][1]  # independent replicas, no shared data


def test_job_throughput_is_summed_over_ranks():
    one = bench.job_tflops(1, 4e12, 2.0)
    assert one == pytest.approx(2000.0)
    assert bench.job_tflops(4, 4e12, 2.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]  # single process: unchanged


def test_reference_arm_does_nothing_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload = bench.DEFAULT_WORKLOAD
        steps = 3
        warmup = 3
        cpu_seconds = 1.0

    assert bench.run_reference(Args) is None
    assert capsys.readouterr().out == ""
