"""The j-slab decomposition of the diffusion (finite_volume_field_gb300/slab.py),
driven on CPU: gloo ranks run the product's slab logic -- slab bounds, halo
bookkeeping, blocks of k steps, step parity, the torch.distributed halo
exchange -- with a CPU stand-in only for the per-slab library call (the
oracle applied to the slab's stored rows with the library's ping-pong
semantics).  The gathered owned rows must equal the single-domain oracle
result bit for bit, for one-row halos (an exchange per step) and for deeper
halos with blocks of several steps (redundant halo rows, one exchange per
block), FP64 and FP32, including slabs of unequal height.
"""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _initial(nx, ny, dt):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from finite_volume_field_gb300 import inputs
    return inputs.diffusion_field(nx, ny, dt, seed=inputs.config_seed(2), stream=5)


def cpu_step(src, dst, nx, ny, alpha, k, dtype, stream):
    """Stand-in for diffuse2d_step on CPU tensors: k steps with the library's
    ping-pong (src -> dst on odd steps) and its result placement."""
    import oracle
    a = src.numpy().reshape(ny, nx)
    b = dst.numpy().reshape(ny, nx)
    u, v, _ = oracle.diffuse2d(a, k, alpha=alpha, v0=b, return_both=True)
    src.copy_(torch.from_numpy(u.reshape(-1)))
    dst.copy_(torch.from_numpy(v.reshape(-1)))


def _worker(rank, world, port, nx, ny, steps, halo, dtname, results):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from finite_volume_field_gb300 import slab
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dt = np.dtype(dtname)
    u0 = _initial(nx, ny, dt)
    rows = slab.slab_rows(ny, world, rank, halo)
    u = torch.from_numpy(u0[rows.l0:rows.l1].reshape(-1).copy())
    v = torch.zeros_like(u)
    s = slab.SlabDiffusion2D(u, v, nx, ny, rows, halo, 0.1, 1 if dt == np.float64 else 0,
                             step=cpu_step)
    s.advance(steps, slab.dist_exchanger(dist, rank, world))
    st = s.state.numpy().reshape(rows.stored, nx)
    results[rank] = st[rows.top:rows.top + (rows.j1 - rows.j0)].copy()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,nx,ny,steps,halo,dt", [
    (2, 37, 29, 9, 1, "float64"),
    (2, 37, 29, 9, 3, "float64"),
    (3, 41, 31, 11, 4, "float32"),
    (3, 16, 26, 7, 8, "float64"),
])
def test_ranks_match_single_domain(world, nx, ny, steps, halo, dt):
    import oracle
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker,
                             args=(r, world, port, nx, ny, steps, halo, dt, results))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
            assert p.exitcode == 0
        glued = np.concatenate([results[r] for r in range(world)], axis=0)
    want = oracle.diffuse2d(_initial(nx, ny, np.dtype(dt)), steps)
    assert glued.shape == want.shape
    assert np.array_equal(glued.view(np.uint8), want.view(np.uint8))


def test_local_slabs_match_single_domain():
    """Several slabs in one process (the one-device form), LocalExchange."""
    import oracle
    from finite_volume_field_gb300 import slab
    nx, ny, steps = 23, 40, 13
    for parts, halo in ((2, 1), (4, 3), (5, 5)):
        u0 = _initial(nx, ny, np.float64)
        slabs = []
        for p in range(parts):
            rows = slab.slab_rows(ny, parts, p, halo)
            u = torch.from_numpy(u0[rows.l0:rows.l1].reshape(-1).copy())
            slabs.append(slab.SlabDiffusion2D(u, torch.zeros_like(u), nx, ny, rows, halo, 0.1, 1,
                                              step=cpu_step))
        slab.LocalExchange(slabs).advance(steps)
        parts_out = []
        for s in slabs:
            r = s.rows
            parts_out.append(s.state.numpy().reshape(r.stored, nx)[r.top:r.top + r.j1 - r.j0])
        got = np.concatenate(parts_out, axis=0)
        want = oracle.diffuse2d(u0, steps)
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64)), (parts, halo)


def test_slab_rows():
    from finite_volume_field_gb300 import slab
    ny = 29
    for parts in (1, 2, 3, 7):
        for halo in (1, 2, 4):
            if parts > 1 and ny // parts < halo:
                with pytest.raises(ValueError):
                    slab.slab_rows(ny, parts, 0, halo)
                continue
            rs = [slab.slab_rows(ny, parts, p, halo) for p in range(parts)]
            assert rs[0].j0 == 0 and rs[-1].j1 == ny
            for a, b in zip(rs, rs[1:]):
                assert a.j1 == b.j0 and a.bottom == b.top == halo
            for r in rs:
                assert r.l0 == max(0, r.j0 - halo) and r.l1 == min(ny, r.j1 + halo)
                assert abs((r.j1 - r.j0) - ny / parts) < 1
