"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2): rank
environment, barrier, max-over-ranks timing and the weak-scaling sum.  The
path itself has no exchange step; this covers only the harness."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    ms = 10.0 + 5.0 * rank                       # per-rank time
    worst = bench.reduce_max(dist, ms, torch.device("cpu"))
    out[rank] = worst
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_max(None, 3.5, torch.device("cpu")) == 3.5
    bench.barrier(None)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_minimum():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
