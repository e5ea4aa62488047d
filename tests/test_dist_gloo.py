"""The N > 1 bench path on CPU: two gloo ranks, no GPU.

Each rank runs an independent chunk (replicas, weak scaling); the only
cross-rank step is the max over ranks of the timed region, and the job's value
counts every rank's pairs.  The reference (oracle) arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 25.0 * rank
    mx = bench.max_over_ranks(local_ms, torch.device("cpu"))
    val = bench.whole_job_value(pairs_per_step=1000, steps=4, world=world, elapsed_ms=mx)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, mx, val))


def test_two_rank_max_and_whole_job_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in res:
        assert mx == 125.0                           # slowest rank
        assert val == pytest.approx(2 * 1000 * 4 / 0.125)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload, dtype, steps, warmup, ref_queries = "1m", "bf16", 1, 0, 1
    assert bench.run_reference(A) == 0              # returns at once, no work
