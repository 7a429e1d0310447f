"""Every entry point through the index-checking debug build (libfvf_check.so,
built with FVF_BOUNDS_CHECK): on small grids that exercise every kernel (the
scalar, march, blocked and both cluster 2D diffusion kernels, both 3D kernels, the
x and transposing packs with and without the copy, the flux difference, the
stage update), the results must still match the oracle bit for bit and no
kernel may have met an index outside its arrays (fvf_device_error bit 2)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    torch = torch_cuda()
    from finite_volume_field_gb300 import buildlib
    path = buildlib.build(bounds_check=True)
    saved = (api.LIB_PATH, api._lib)
    api.LIB_PATH, api._lib = path, None
    api.load()
    assert api.device_error() == 0
    yield torch
    api.LIB_PATH, api._lib = saved


def _no_flags():
    assert api.device_error() == 0, "a kernel met an out-of-range index (or a wait expired)"


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("nx,ny,steps", [
    (31, 27, 7), (3, 5, 2),                 # 8-block cluster kernel (all steps in one launch)
    (64, 64, 32), (33, 65, 5),               # 16-block cluster kernel
    (2048, 200, 9),                          # FP32: blocked kernel, then one single step
    (2048, 200, 1),                          # vector march kernel
    (2047, 100, 1),                          # scalar kernel (rows not 16-byte aligned)
])
def test_diffusion_2d_checked(checked, dt, nx, ny, steps):
    torch = checked
    u0 = inputs.diffusion_field(nx, ny, dt, seed=inputs.config_seed(2))
    u, v = to_dev(u0), torch.zeros(u0.size, dtype=u_dtype(torch, dt), device="cuda")
    api.diffuse2d_step(u, v, nx, ny, 0.1, steps)
    torch.cuda.synchronize()
    want = oracle.diffuse2d(u0.reshape(ny, nx), steps)
    assert_bits_equal(to_host(v if steps % 2 else u), want)
    _no_flags()


def u_dtype(torch, dt):
    return torch.float64 if dt == np.float64 else torch.float32


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("shape", [(9, 10, 12), (5, 6, 7), (40, 9, 64), (12, 25, 66)])
def test_diffusion_3d_checked(checked, dt, shape):
    torch = checked
    u0 = inputs.uniform_f64(41, 0, int(np.prod(shape))).reshape(shape).astype(dt)
    u = to_dev(u0.reshape(-1))
    v = torch.zeros_like(u)
    nz, ny, nx = shape
    api.diffuse3d_step(u, v, nx, ny, nz, 0.1, 3)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(v).reshape(shape), oracle.diffuse3d(u0, 3, 0.1))
    _no_flags()


@pytest.mark.parametrize("extents,g", [((5, 4, 3), 2), ((33, 31, 35), 3), ((65, 66, 1), 2)])
def test_pack_copy_flux_stage_checked(checked, extents, g):
    torch = checked
    nv = 3
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    dev = [to_dev(f) for f in fields]
    for direction in range(3):
        M = oracle.pack_extents(extents, g, direction)
        out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float64, device="cuda")
        api.weno_pack(dev, nv, extents, g, direction, out)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(out), oracle.weno_pack(fields, extents, g, direction))
        copies = [torch.empty_like(d) for d in dev]
        api.weno_pack_copy(dev, nv, extents, g, direction, out, copies)
        torch.cuda.synchronize()
        want_pack, want_copies = oracle.weno_pack_copy(fields, extents, g, direction)
        assert_bits_equal(to_host(out), want_pack)
        for c, w in zip(copies, want_copies):
            assert_bits_equal(to_host(c), w)
        f32 = [f.astype(np.float32) for f in fields]
        o32 = torch.empty(out.numel(), dtype=torch.float32, device="cuda")
        api.weno_pack_f32([to_dev(f) for f in f32], nv, extents, g, direction, o32)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(o32), oracle.weno_pack(f32, extents, g, direction))
    copies = [torch.empty_like(d) for d in dev]
    api.fields_copy(dev, nv, extents, g, copies)
    torch.cuda.synchronize()
    for c, f in zip(copies, fields):
        assert_bits_equal(to_host(c), f)
    seed = inputs.config_seed(4)
    n = int(np.prod(extents)) * nv
    fl = [inputs.face_fluxes(seed, nv, extents, d) for d in range(3)]
    w = [inputs.inverse_spacing(seed, extents[d], stream=200 + d) for d in range(3)]
    rhs = torch.empty(n, dtype=torch.float64, device="cuda")
    want = None
    for d in range(3):
        fn = api.advect_rhs if d == 0 else api.advect_rhs_add
        fn(to_dev(fl[d]), to_dev(w[d]), nv, extents, d, rhs)
        torch.cuda.synchronize()
        want = (oracle.advect_rhs(fl[d], w[d], nv, extents, d) if d == 0
                else oracle.advect_rhs_add(fl[d], w[d], nv, extents, d, want))
        assert_bits_equal(to_host(rhs), want)
        sweep = torch.empty(fl[d].size, dtype=torch.float64, device="cuda")
        api.flux_unpack(to_dev(fl[d]), nv, extents, d, sweep)
        torch.cuda.synchronize()
    r32 = torch.empty(n, dtype=torch.float32, device="cuda")
    api.advect_rhs_f32(to_dev(fl[1].astype(np.float32)), to_dev(w[1].astype(np.float32)), nv,
                       extents, 1, r32)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(r32), oracle.advect_rhs(fl[1].astype(np.float32),
                                                      w[1].astype(np.float32), nv, extents, 1))
    u0, u1 = inputs.normal_f64(5, 0, n), inputs.normal_f64(5, 1, n)
    out = torch.empty(n, dtype=torch.float64, device="cuda")
    api.ssprk3_stage(to_dev(u0), to_dev(u1), [to_dev(f) for f in fl], [to_dev(x) for x in w], nv,
                     extents, 0.75, 0.25, 0.1, out)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(out), oracle.ssprk3_stage(u0, u1, fl, w, nv, extents, 0.75, 0.25, 0.1))
    api.ssprk3_axpby(to_dev(u0), to_dev(u1), rhs, nv, extents, 1.0 / 3.0, 2.0 / 3.0, 0.1, out)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(out), oracle.rk_axpby(u0, u1, want, 1.0 / 3.0, 2.0 / 3.0, 0.1))
    _no_flags()
