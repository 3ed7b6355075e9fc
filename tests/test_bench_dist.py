"""The benchmark's multi-rank plumbing on CPU with gloo, world size 2: every
rank reaches the barrier and the reported time is the slowest rank's."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist = bench.init_dist(ws, "gloo")
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 10.0 + rank)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (1, 0, 0)
    assert bench.init_dist(ws, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_reference_arm_reports_on_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.main.__globals__["argparse"].Namespace(steps=1, warmup=0)) is None
    assert capsys.readouterr().out == ""
