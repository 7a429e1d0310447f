"""The j-slab decomposition on one device through the library (slab.py with
LocalExchange: halo rows copied between slabs, every step in diffuse2d_step's
kernels), against the single-domain oracle: the full 8192 x 8192, 200-step
workload in two slabs (FP64 with 4-row halos, FP32 with 8-row halos so that
each block of 8 steps takes the shared-memory blocked kernel), and ragged
grids in three slabs."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs, slab
from tests.gpu_util import assert_bits_equal, torch_cuda

pytestmark = pytest.mark.gpu


def _run_slabs(torch, u0: np.ndarray, steps: int, parts: int, halo: int):
    ny, nx = u0.shape
    code = api.FVF_FP64 if u0.dtype == np.float64 else api.FVF_FP32
    slabs = []
    for p in range(parts):
        rows = slab.slab_rows(ny, parts, p, halo)
        u = torch.from_numpy(u0[rows.l0:rows.l1].reshape(-1).copy()).to("cuda")
        slabs.append(slab.SlabDiffusion2D(u, torch.zeros_like(u), nx, ny, rows, halo, 0.1, code))
    slab.LocalExchange(slabs).advance(steps)
    torch.cuda.synchronize()
    out = []
    for s in slabs:
        r = s.rows
        out.append(s.state.cpu().numpy().reshape(r.stored, nx)[r.top:r.top + r.j1 - r.j0])
    return np.concatenate(out, axis=0)


@pytest.mark.parametrize("dt,halo", [(np.float64, 4), (np.float32, 8)])
def test_two_slabs_full_size(dt, halo):
    torch = torch_cuda()
    n = 8192
    u0 = inputs.diffusion_field(n, n, dt, seed=inputs.config_seed(2),
                                stream=0 if dt == np.float32 else 1)
    got = _run_slabs(torch, u0, 200, 2, halo)
    want = oracle.diffuse2d(u0, 200, nthreads=oracle.max_threads())
    assert_bits_equal(got, want, what=f"two slabs 8192^2 {dt.__name__}")


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("nx,ny,steps,halo", [(1000, 307, 23, 3), (258, 96, 17, 8), (77, 60, 9, 1)])
def test_three_slabs_ragged(dt, nx, ny, steps, halo):
    torch = torch_cuda()
    n = nx * ny
    u0 = (inputs.uniform_f32(13, nx + ny, n) if dt == np.float32
          else inputs.uniform_f64(13, nx + ny, n)).reshape(ny, nx)
    u0[0, :] = 0
    u0[-1, :] = 0
    got = _run_slabs(torch, u0, steps, 3, halo)
    assert_bits_equal(got, oracle.diffuse2d(u0, steps), what=f"{nx}x{ny} {steps} halo {halo}")
