"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
runs its own replica, the step time is the max over ranks, the whole-job rate
counts the units of all ranks, and the reference arm runs on rank 0 only."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [12.5, 20.0][rank]
    ms = bench.job_time_ms(local, world)
    rate = bench.whole_job_rate(1000, world, ms)
    w, r, lr = bench.dist_env()
    out.put((rank, ms, rate, w, r, lr))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_max_time_and_rate():
    import random
    port = 29500 + random.randint(0, 2000)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, w, r, lr in res:
        assert ms == 20.0
        assert rate == pytest.approx(2 * 1000 / 0.020)
        assert (w, r, lr) == (2, rank, rank)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(7.0, 1) == 7.0
    assert bench.whole_job_rate(131072, 1, 1000.0) == pytest.approx(131072.0)


def test_reference_arm_other_ranks_exit(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from sparse_attention_kpool_compress_gb300 import workloads as W
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, ref_rows = 1, 3, 4
    assert bench.run_reference(A(), W.WORKLOADS["tiny"]) == 0
