"""The multi-rank host logic of bench.py on CPU: two gloo ranks agree on the slowest
rank's step time and on the whole-job (weak-scaling) throughput; a batch split by
sequence across the ranks (the partition bench.py runs for N > 1) gives, rank by rank,
exactly the rows of the whole batch; and the reference arm runs on rank 0 only."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
import synth


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


def _shard_main(rank, world, port, name, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shard = synth.workload_shard(name, rank, world)
        o, lse = oracle.full(shard, threads=2)
        got = [None] * world
        dist.all_gather_object(got, (list(synth.shard_sequences(shard.batch * world, rank, world)), o, lse))
        out[rank] = got
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny_mqa_decode"])
def test_batch_split_by_sequence_over_two_gloo_ranks(name):
    """Each rank builds and runs (in the oracle) its shard of the global batch; gathered,
    the shards' rows are the whole batch's rows, sequence for sequence."""
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_shard_main, args=(world, port, name, out), nprocs=world, join=True)
    got = out[0]
    assert [g[0] for g in got] == [g[0] for g in out[1]]  # every rank gathered the same shards
    ids = [b for g in got for b in g[0]]
    per = synth.WORKLOADS[name]["batch"]
    assert ids == list(range(per * world))  # a partition of the global batch, in order
    whole = synth.concat_cases([synth.workload_shard(name, r, world) for r in range(world)])
    o_all, lse_all = oracle.full(whole)
    qo = whole.qo_indptr.tolist()
    for seqs, o, lse in got:
        rows = [t for b in seqs for t in range(qo[b], qo[b + 1])]
        assert np.array_equal(o_all[rows], o) and np.array_equal(lse_all[rows], lse)


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
