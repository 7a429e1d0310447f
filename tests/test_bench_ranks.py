"""The benchmark's multi-rank host logic, run as two gloo ranks on the CPU.

Each rank is an independent replica of the whole workload; the process group
only carries the timing barrier and the gather of per-rank results.  Here
each rank contributes made-up per-rank timings, gathers them with
all_gather_object exactly as bench.py does, and rank 0 checks the
aggregation (device time = max over ranks, launches = sum).  The reference
arm's non-zero ranks must exit without doing any work.
"""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = {"ms_per_step": 10.0 + 5.0 * rank, "e2e_ms_per_step": 20.0 - rank,
            "launches": 806 + rank}
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    ms, e2e_ms, launches = bench.aggregate(gathered, world)
    dist.barrier()
    dist.destroy_process_group()
    # The reference arm: every rank but 0 returns at once, before any work.
    ref_rc = bench.run_reference(bench.argparse.Namespace(steps=1, warmup=0, gpus=world)) \
        if rank != 0 else 0
    results[rank] = (ms, e2e_ms, launches, ref_rc)


def test_two_rank_aggregation():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    for rank in range(world):
        ms, e2e_ms, launches, ref_rc = res[rank]
        assert ms == 15.0          # max over ranks
        assert e2e_ms == 20.0      # max over ranks
        assert launches == 806 + 807
        assert ref_rc == 0
