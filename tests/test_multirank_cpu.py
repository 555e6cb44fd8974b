"""The N > 1 host path of bench.py on CPU: two gloo ranks.

Every (document, head) and every (sequence, KV head) is independent, so the
GPUs run independent weak-scaled replicas; the only collectives are the
barrier and the max / sum over ranks of the timings and work counts.  These
tests run those host functions as two processes on the gloo backend."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # a rank's own timing and work; the job reports the slowest rank's time
    ms = 2.0 + rank  # rank 1 is slower
    work = 100.0 * (rank + 1)
    mx = bench.max_over_ranks(ms, w)
    tot = bench.sum_over_ranks(work, w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{mx} {tot}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        mx, tot = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert mx == 3.0  # max over ranks: the job is as slow as its slowest replica
        assert tot == 300.0  # whole-job work: both replicas' work counted


def test_single_rank_reductions_are_identity(monkeypatch):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(1) == (1, 0, 0)
    assert bench.max_over_ranks(1.5, 1) == 1.5 and bench.sum_over_ranks(7.0, 1) == 7.0
