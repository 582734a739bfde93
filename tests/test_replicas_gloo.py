"""The N-replica path of bench.py on CPU: two gloo ranks (no GPU).

Every rank runs an independent replica and nothing is exchanged on the data
path; the only collective is the timing reduction (the slowest rank sets the
job time) and the barriers around the timed region.  The reference arm runs
on rank 0 alone.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._dist = dist
    try:
        bench.barrier()
        got = bench.max_over_ranks(1.5 + rank)  # per-rank "times"
        bench.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()
        bench._dist = None


def test_two_gloo_ranks_reduce_to_the_slowest():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"workload": "tiny_causal", "steps": 1, "warmup": 0, "ref_budget": 0.1})()
    bench.run_reference(args)  # a non-zero rank returns at once and prints nothing
    assert capsys.readouterr().out == ""
