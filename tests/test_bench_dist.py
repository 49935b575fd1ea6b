"""The multi-rank timing logic of bench.py on CPU: two gloo ranks, each with
its own batch (weak scaling); the job time is the max over ranks and the work
is the sum (no collective on the data path)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), SPECDEC_BENCH_BACKEND="gloo")
    import torch.distributed as dist

    import bench

    r, local, w, _ = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    secs, units = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), w)
    bench.barrier(w)
    q.put((rank, secs, units))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for _, secs, units in res:
        assert secs == 2.0 and units == 300.0


def test_reference_arm_runs_only_on_rank_zero(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
