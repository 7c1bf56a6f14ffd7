"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun every rank runs its own batch of the workload on its own GPU
(independent sequences, no data-path collective); the only cross-rank steps
are the barrier around the timed region and the max over ranks of the time.
These tests run that host logic with the gloo backend, without a GPU.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import m3synth  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.distributed.barrier()
        ms = bench.max_over_ranks(torch, times[rank], world, torch.device("cpu"))
        idx, shape = m3synth.WORKLOADS["tiny"]
        inp = m3synth.scan_inputs(shape, seed=bench.rank_seed(idx, rank))
        q.put((rank, ms, bench.job_rate(shape.tokens, world, ms),
               float(np.asarray(inp["x"], np.float64).sum())))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job_rate():
    world, times = 2, [0.25, 0.31]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    tokens = m3synth.WORKLOADS["tiny"][1].tokens
    for rank, ms, rate, _ in res:
        assert ms == pytest.approx(max(times))  # every rank gets the slowest time
        assert rate == pytest.approx(world * tokens / (max(times) * 1e-3))
    # weak scaling: each rank draws its own batch
    assert res[0][3] != res[1][3]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, 0.5, 1, torch.device("cpu")) == 0.5
    assert bench.job_rate(1000, 1, 2.0) == pytest.approx(500000.0)
    assert bench.rank_seed(3, 0) == 3 and bench.rank_seed(3, 1) != 3


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
