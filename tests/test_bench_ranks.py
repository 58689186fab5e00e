"""The benchmark's replica timing on several processes (gloo on CPU, world
size 2): every rank sees the slowest rank's time, and the whole-job value
counts all ranks' steps over it."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
    slowest = b.slowest_rank_ms(mine, torch.device("cpu"), dist)
    out[rank] = (slowest, b.whole_job_tflops(world, 4, 1e12, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_and_whole_job_value():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, value = out[0]
    assert slowest == pytest.approx(15.0)
    # 2 ranks x 4 steps x 1e12 flops in 15 ms
    assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_needs_no_group():
    b = _bench()
    assert b.slowest_rank_ms(7.5, torch.device("cpu"), None) == 7.5
    assert b.whole_job_tflops(1, 10, 2e12, 20.0) == pytest.approx(1000.0)
