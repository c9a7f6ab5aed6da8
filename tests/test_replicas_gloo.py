"""The N > 1 path of bench.py on CPU: two `gloo` ranks run the timing reduction the
GPU replicas use (barrier, slowest rank's time, whole-job tokens/s), and the
reference arm's non-zero ranks leave without work."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    ms = bench.slowest_ms(100.0 + 25.0 * rank, world, "cpu")  # rank 1 is the slow one
    out[rank] = (ms, bench.job_throughput(32768, world, 10, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 125.0
    assert value == pytest.approx(32768 * 2 * 10 / 0.125)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_ms(42.0, 1, "cpu") == 42.0
    assert bench.job_throughput(100, 1, 4, 2000.0) == pytest.approx(200.0)


def test_reference_arm_non_zero_rank_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        config, shape, chunk, steps, warmup, ref_rows = 3, None, 0, 1, 0, 1

    assert bench.run_reference(Args()) == 0
