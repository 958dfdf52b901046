"""The benchmark's N > 1 path (replicas): two ranks on the CPU with gloo. The job's
time is the slowest rank's, its rate the units of all ranks over that time."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_of_rank, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max = bench.slowest_rank_ms(ms_of_rank[rank], torch.device("cpu"))
        rate = bench.whole_job_rate(150e6, 100, world, ms_max)
        out[rank] = (ms_max, rate)
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    ms_of_rank = [10.0, 12.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), ms_of_rank, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms_max, rate = res[r]
        assert ms_max == 12.5
        assert rate == pytest.approx(150e6 * 100 * 2 / 12.5e-3)


def test_single_rank_without_process_group():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.slowest_rank_ms(7.0, torch.device("cpu")) == 7.0
    assert bench.whole_job_rate(1e9, 10, 1, 1000.0) == pytest.approx(1e10)
