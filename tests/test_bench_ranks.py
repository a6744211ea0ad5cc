"""The bench's cross-rank logic with two gloo ranks on the CPU.

`bench.py --gpus N` runs one replica per rank (weak scaling, no data-path
exchange); its value is all ranks' units over the slowest rank's time. These
tests run that aggregation, as bench.py calls it, in two CPU processes.
"""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        local = [2.0, 3.5][rank]                 # each rank's own time
        t_max = b.max_over_ranks(local, "cpu", world)
        rate = b.whole_job_rate(100.0, 10, world, t_max)
        out[rank] = (t_max, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_units():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        assert out[0] == out[1]
        t_max, rate = out[0]
        assert t_max == 3.5
        assert rate == pytest.approx(2 * 100.0 * 10 / 3.5)


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(1.25, "cpu", 1) == 1.25
    assert b.whole_job_rate(10.0, 4, 1, 2.0) == 20.0
