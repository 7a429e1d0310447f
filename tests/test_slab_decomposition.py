"""The multi-GPU decomposition of the diffusion sweep, checked on CPU ranks.

Two gloo ranks each own a band of rows (a slab along j) plus one halo row on
the side facing the other rank.  Every step each rank applies the update to
its slab with the CPU oracle, then the ranks swap the rows next to the cut
(nx values each way).  After n steps the gathered slabs must equal the
single-domain result bit for bit: the update of a cell reads only its four
neighbours, so one halo row per step is the whole exchange, and no
collective other than that neighbour send/recv is needed.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

NX, NY, CUT, STEPS = 37, 29, 13, 9


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _initial():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from finite_volume_field_gb300 import inputs
    return inputs.diffusion_field(NX, NY, np.float64, seed=inputs.config_seed(2), stream=5)


def _worker(rank, port, results):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    u0 = _initial()
    # rank 0: global rows [0, CUT] (row CUT is its halo); rank 1: rows [CUT-1, NY) (row CUT-1 halo)
    local = u0[: CUT + 1].copy() if rank == 0 else u0[CUT - 1:].copy()
    for _ in range(STEPS):
        local = oracle.diffuse2d(local, 1)
        if rank == 0:
            send, recv_into = local[CUT - 1], CUT       # last owned row -> rank 1's halo
        else:
            send, recv_into = local[1], 0               # first owned row -> rank 0's halo
        buf = torch.empty(NX, dtype=torch.float64)
        ops = [dist.P2POp(dist.isend, torch.from_numpy(send.copy()), 1 - rank),
               dist.P2POp(dist.irecv, buf, 1 - rank)]
        for r in dist.batch_isend_irecv(ops):
            r.wait()
        local[recv_into] = buf.numpy()
    owned = local[:CUT] if rank == 0 else local[1:]
    results[rank] = owned.copy()
    dist.barrier()
    dist.destroy_process_group()


def test_two_slabs_match_single_domain():
    import oracle
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        glued = np.concatenate([results[0], results[1]], axis=0)
    want = oracle.diffuse2d(_initial(), STEPS)
    assert glued.shape == want.shape
    assert np.array_equal(glued.view(np.uint64), want.view(np.uint64))
