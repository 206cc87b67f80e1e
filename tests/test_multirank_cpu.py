"""The benchmark's multi-rank path on CPU with gloo, world size 2: every rank
reads its place from the launcher's environment, the reported time is the
slowest rank's, and the reference arm runs on rank 0 only.  (The decode path
itself runs as independent replicas, one per GPU, with no collective.)"""
import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.rank_env()
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        q.put((rank, env, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for rank, env, got in res:
        assert env == (2, rank, rank)
        assert got == 15.0  # the slower rank's time on every rank


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(gpus=2, steps=2, warmup=3, impl="reference", workload="qwen3_8b_100k", cpu_budget=1.0)
    assert bench.run_reference(args, bench.WORKLOADS["qwen3_8b_100k"]) is None
    assert capsys.readouterr().out == ""
