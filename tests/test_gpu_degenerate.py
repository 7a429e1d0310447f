"""GPU results of the degenerate sizes the boundary accepts (include/fvf.h):
a grid with no interior gets zeros written to its destination every step;
empty grids, nv = 0 and zero extents leave every buffer untouched and launch
nothing; a swept axis of extent 1 (a 2D field swept along z) packs and
differences exactly as the oracle's definition does."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

DT = {np.float32: api.FVF_FP32, np.float64: api.FVF_FP64}


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("nx,ny", [(1, 1), (2, 2), (2, 9), (9, 2), (1, 12), (12, 1)])
def test_no_interior_grid_writes_zeros(dt, nx, ny):
    torch = torch_cuda()
    u0 = (inputs.uniform_f64(31, nx + 100 * ny, nx * ny) + 1.0).astype(dt).reshape(ny, nx)
    v0 = (inputs.uniform_f64(32, nx + 100 * ny, nx * ny) + 1.0).astype(dt).reshape(ny, nx)
    for steps, zero_u, zero_v in ((1, False, True), (2, True, True), (3, True, True)):
        u, v = to_dev(u0), to_dev(v0)
        api.diffuse2d_step(u, v, nx, ny, 0.1, steps, DT[dt])
        torch.cuda.synchronize()
        gu, gv = to_host(u).reshape(ny, nx), to_host(v).reshape(ny, nx)
        assert_bits_equal(gu, np.zeros_like(u0) if zero_u else u0, what=f"u {steps}")
        assert_bits_equal(gv, np.zeros_like(v0) if zero_v else v0, what=f"v {steps}")
        ou, ov, _ = oracle.diffuse2d(u0, steps, v0=v0, return_both=True)
        assert_bits_equal(gu, ou, what="u vs oracle")
        assert_bits_equal(gv, ov, what="v vs oracle")


def test_empty_calls_touch_nothing():
    torch = torch_cuda()
    u = torch.full((64,), 7.0, dtype=torch.float64, device="cuda")
    v = torch.full((64,), 9.0, dtype=torch.float64, device="cuda")
    before = api.launch_count()
    api.diffuse2d_step(u, v, 8, 8, 0.1, 0, api.FVF_FP64)       # nsteps 0
    api.diffuse2d_step(u, v, 0, 8, 0.1, 4, api.FVF_FP64)       # empty grid
    api.diffuse3d_step(u, v, 4, 4, 0, 0.1, 4, api.FVF_FP64)    # empty 3D grid
    out = torch.full((64,), 5.0, dtype=torch.float64, device="cuda")
    api.weno_pack([u], 0, (4, 4, 4), 0, 0, out)               # nv 0
    api.weno_pack([u], 1, (4, 0, 4), 0, 1, out)               # a zero extent
    api.advect_rhs(u, v, 0, (2, 2, 2), 0, out)                # nv 0
    api.advect_rhs_add(u, v, 1, (0, 2, 2), 1, out)            # a zero extent
    api.flux_unpack(u, 0, (2, 2, 2), 2, out)
    torch.cuda.synchronize()
    assert api.launch_count() == before
    assert bool((u == 7.0).all()) and bool((v == 9.0).all()) and bool((out == 5.0).all())


@pytest.mark.parametrize("dt", [np.float64, np.float32])
def test_pack_along_axis_of_extent_one(dt):
    """A 2D field (n3 = 1: stored N3 = 1, no ghosts on that axis) packed
    along z: the packed output has extent 1 on the swept axis."""
    torch = torch_cuda()
    ext, g, nv = (6, 5, 1), 2, 3
    fields = [f.astype(dt) for f in inputs.normal_fields(41, nv, ext, g)]
    M = (1, ext[1], ext[0])
    out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float64 if dt == np.float64 else
                      torch.float32, device="cuda")
    f = api.weno_pack if dt == np.float64 else api.weno_pack_f32
    f([to_dev(x) for x in fields], nv, ext, g, 2, out)
    torch.cuda.synchronize()
    want = oracle.weno_pack(fields, ext, g, 2)
    assert_bits_equal(to_host(out), np.asarray(want).reshape(-1), what="pack z, n3 = 1")


def test_flux_difference_along_axis_of_extent_one():
    """advect_rhs along z with n3 = 1: two faces per column,
    rhs = inv_d(0) * (F(-1) - F(0))."""
    torch = torch_cuda()
    ext, nv = (7, 5, 1), 2
    F = inputs.face_fluxes(43, nv, ext, 2)
    w = inputs.inverse_spacing(43, 1)
    rhs = torch.empty(7 * 5 * nv, dtype=torch.float64, device="cuda")
    api.advect_rhs(to_dev(F), to_dev(w), nv, ext, 2, rhs)
    torch.cuda.synchronize()
    want = oracle.advect_rhs(F, w, nv, ext, 2)
    assert_bits_equal(to_host(rhs), np.asarray(want).reshape(-1), what="rhs z, n3 = 1")
