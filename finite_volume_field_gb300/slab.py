"""Slab decomposition of the 2D diffusion along j (rows), with halo rows.

The grid's ny rows are split into ``parts`` slabs of near-equal height; slab
p owns rows [j0, j1) and stores rows [l0, l1) = its owned rows plus up to
``halo`` rows on each side (clipped to the grid), full width.  A slab
advances ``k <= halo`` steps at a time with the library's own
``diffuse2d_step`` on its stored rows (FP32 then takes the shared-memory
blocked kernel for k > 2), then exchanges halos: it sends its first and last
``halo`` owned rows to its neighbours and receives theirs into its halo
rows.  One exchange per ``k`` steps (halos as deep as the block of steps,
as in temporal blocking; with k = 1, one row per step).

Why this reproduces the single-grid result bit for bit: the library treats
the first and last stored rows as edges and writes zeros there each step.
For an inner slab those rows are halo rows, not global edges, so their
values are wrong after the first local step, and the error moves one row
inward per step.  After k <= halo steps it has reached at most halo - 1 rows
in from the stored edge: the owned rows (at distance >= halo) are exact, and
the halos are refreshed by the exchange before the next block.  The slabs at
the top and bottom of the grid store the real edge rows, which the library
zeroes as the single grid does; the two column edges are global edges of
every slab.

Only rows cross between parts, and a row is contiguous (column-major, i
fastest), so an exchange is two sends and two receives of halo*nx elements
per neighbour.  The exchange is an object with one method (``DistExchange``:
torch.distributed point-to-point between ranks; ``LocalExchange``: copies
between slabs held by one process), so the same host logic drives one slab
per GPU and several slabs on one device.  Every step of the arithmetic runs
in the library's kernels (``step`` may be replaced only by tests that stand
in for the device).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class SlabRows:
    """Rows of one slab: owned [j0, j1), stored [l0, l1), both global."""
    j0: int
    j1: int
    l0: int
    l1: int

    @property
    def stored(self) -> int:
        return self.l1 - self.l0

    @property
    def top(self) -> int:
        """Halo rows stored below the owned rows (rows l0 .. j0-1)."""
        return self.j0 - self.l0

    @property
    def bottom(self) -> int:
        """Halo rows stored above the owned rows (rows j1 .. l1-1)."""
        return self.l1 - self.j1


def slab_rows(ny: int, parts: int, index: int, halo: int) -> SlabRows:
    """Owned and stored rows of slab ``index`` of ``parts`` slabs of a grid of
    ``ny`` rows, ``halo`` halo rows each side.  Slab heights differ by at most
    one row; every slab must own at least ``halo`` rows (so that a halo comes
    from the adjacent slab alone) unless there is one slab."""
    if parts < 1 or not 0 <= index < parts:
        raise ValueError("need 0 <= index < parts")
    if halo < 1:
        raise ValueError("halo must be >= 1")
    base, extra = divmod(ny, parts)
    if parts > 1 and base < halo:
        raise ValueError(f"{ny} rows in {parts} slabs leave fewer than {halo} rows per slab")
    j0 = index * base + min(index, extra)
    j1 = j0 + base + (1 if index < extra else 0)
    return SlabRows(j0, j1, max(0, j0 - halo), min(ny, j1 + halo))


class DistExchange:
    """Halo exchange between ranks with torch.distributed point-to-point
    (NCCL between GPUs, gloo between CPU processes): slab p is rank p."""

    def __init__(self, dist, rank: int, world: int, group=None):
        self.dist, self.rank, self.world, self.group = dist, rank, world, group

    def exchange(self, sends: dict, recvs: dict) -> None:
        """sends/recvs map a neighbour offset (-1: the slab below, +1: the one
        above) to a contiguous tensor; matching sizes on both sides."""
        ops = []
        for off, t in sends.items():
            ops.append(self.dist.P2POp(self.dist.isend, t, self.rank + off, self.group))
        for off, t in recvs.items():
            ops.append(self.dist.P2POp(self.dist.irecv, t, self.rank + off, self.group))
        if ops:
            for req in self.dist.batch_isend_irecv(ops):
                req.wait()


class SlabDiffusion2D:
    """One slab of a j-decomposed 2D diffusion (u, v: its stored rows, flat
    column-major tensors of rows.stored * nx elements; u holds the current
    state on entry).  ``advance`` runs steps in blocks of at most ``halo``,
    exchanging halos before each block; ``state`` is the buffer holding the
    latest state."""

    def __init__(self, u, v, nx: int, ny: int, rows: SlabRows, halo: int, alpha: float,
                 dtype: int, stream=None, step=None):
        from . import api
        self.u, self.v = u, v
        self.nx, self.ny, self.rows, self.halo = nx, ny, rows, halo
        self.alpha, self.dtype, self.stream = alpha, dtype, stream
        self.step = step if step is not None else api.diffuse2d_step
        self.cur = 0          # 0: state in u, 1: state in v

    @property
    def state(self):
        return self.u if self.cur == 0 else self.v

    def _rows(self, buf, first: int, count: int):
        """View of `count` stored rows starting at global row `first`."""
        a = (first - self.rows.l0) * self.nx
        return buf[a:a + count * self.nx]

    def halo_buffers(self):
        """(sends, recvs) of the current state for an exchange: the first and
        last ``halo`` owned rows go to the slab below / above; the halo rows
        are received.  Sends are views of owned rows, receives views of halo
        rows of the same buffer (disjoint)."""
        r, h, s = self.rows, self.halo, self.state
        sends, recvs = {}, {}
        if r.top:
            sends[-1] = self._rows(s, r.j0, r.top)
            recvs[-1] = self._rows(s, r.l0, r.top)
        if r.bottom:
            sends[+1] = self._rows(s, r.j1 - r.bottom, r.bottom)
            recvs[+1] = self._rows(s, r.j1, r.bottom)
        return sends, recvs

    def local_steps(self, k: int) -> None:
        """k steps of the library on the stored rows (k <= halo)."""
        if k < 1:
            return
        src, dst = (self.u, self.v) if self.cur == 0 else (self.v, self.u)
        self.step(src, dst, self.nx, self.rows.stored, self.alpha, k, self.dtype, self.stream)
        if k % 2:
            self.cur ^= 1

    def advance(self, nsteps: int, exchange) -> None:
        """nsteps steps: blocks of at most ``halo`` steps, each preceded by a
        halo exchange (``exchange(slab)`` performs it for this slab)."""
        done = 0
        while done < nsteps:
            k = min(self.halo, nsteps - done)
            exchange(self)
            self.local_steps(k)
            done += k


def dist_exchanger(dist, rank: int, world: int, group=None, sync=None):
    """An ``exchange(slab)`` callable for ``SlabDiffusion2D.advance`` on one
    rank: the slab's halos with its neighbours over torch.distributed.
    ``sync`` (e.g. a stream synchronisation) runs before the sends, so that
    the rows sent are the finished state."""
    ex = DistExchange(dist, rank, world, group)

    def exchange(slab):
        if sync is not None:
            sync()
        sends, recvs = slab.halo_buffers()
        ex.exchange({o: t.contiguous() for o, t in sends.items()}, recvs)
    return exchange


class LocalExchange:
    """Halo exchange among the slabs of one process (e.g. several slabs on
    one device): copies each slab's boundary owned rows into its
    neighbours' halo rows.  All slabs advance together: ``advance`` runs
    each block on every slab, exchanging first."""

    def __init__(self, slabs):
        self.slabs = list(slabs)

    def exchange_all(self) -> None:
        bufs = [s.halo_buffers() for s in self.slabs]
        for p, (sends, _) in enumerate(bufs):
            for off, t in sends.items():
                bufs[p + off][1][-off].copy_(t)

    def advance(self, nsteps: int) -> None:
        halo = min(s.halo for s in self.slabs)
        done = 0
        while done < nsteps:
            k = min(halo, nsteps - done)
            self.exchange_all()
            for s in self.slabs:
                s.local_steps(k)
            done += k
