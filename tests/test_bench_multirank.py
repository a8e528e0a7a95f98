"""The multi-rank host logic of bench.py on CPU: two gloo ranks agree on the slowest
rank's step time and on the whole-job (weak-scaling) throughput, and the reference arm
runs on rank 0 only."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.0 + rank * 0.5  # rank 1 is the slower one
        slowest = bench.max_over_ranks(ms, device="cpu")
        value = bench.weak_scaling_value(2.0e9, world, slowest)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of this (threaded) process
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 1.5
        # 2 GB per rank, two ranks, 1.5 ms: 2666.67 GB/s for the job
        assert value == pytest.approx(2.0e9 * 2 / 1.5e-3 / 1e9)


def test_without_a_group_the_local_time_is_used():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25, device="cpu") == 3.25
    assert bench.weak_scaling_value(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""


def test_source_digest_ignores_comments_not_code():
    base = 'int f(int x) { return x + 1; }  // add one\n/* block */ const char* s = "a // b";\n'
    same = '// header\nint f(int x) {\n  return x + 1;  /* changed comment */\n}\nconst char* s = "a // b";\n'
    other = 'int f(int x) { return x + 2; }\nconst char* s = "a // b";\n'
    lit = 'int f(int x) { return x + 1; }\nconst char* s = "a // c";\n'
    d = lambda t: bench.sources_digest(["x.cu"], read=lambda n: t)
    assert d(base) == d(same)
    assert d(base) != d(other) and d(base) != d(lit)
