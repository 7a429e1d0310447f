"""Grids of more than 2^31 elements, where any 32-bit index arithmetic would
wrap: the 2D diffusion (blocked kernel, FP32), the 3D diffusion (bulk-copy
kernel, FP32) and the x and z packs (FP64), checked at sampled outputs.

A diffusion cell after s steps depends only on the (2s+1)^2 (2D) or
(2s+1)^3 (3D) cells around it, so the oracle runs on that window cut from the
initial field (its own edge rule only touches cells the centre no longer
depends on) and its centre value must equal the GPU's bit for bit.  The pack
is checked against its defining index mapping on values built from the
element index."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bits_equal, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def _ramp(torch, n, mod, off, scale, dtype):
    t = torch.arange(n, dtype=torch.float64, device="cuda")
    return t.remainder_(mod).sub_(off).mul_(scale).to(dtype)


def test_diffusion_2d_fp32_beyond_2_31_cells():
    torch = torch_cuda()
    from finite_volume_field_gb300 import api
    nx, ny, steps = 65536, 32770, 3          # 2.15e9 cells, 8.6 GB per buffer
    n = nx * ny
    u = _ramp(torch, n, 1000003.0, 0.0, 1e-6, torch.float32)
    v = torch.zeros_like(u)
    api.diffuse2d_step(u, v, nx, ny, 0.1, steps, api.FVF_FP32)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    rng = np.random.default_rng(7)
    pts = np.stack([rng.integers(steps, nx - steps, 64), rng.integers(steps, ny - steps, 64)], 1)
    pts = np.concatenate([pts, [[steps, steps], [nx - 1 - steps, ny - 1 - steps],
                                [nx // 2, ny - 1 - steps]]])
    u0 = _ramp(torch, n, 1000003.0, 0.0, 1e-6, torch.float32).view(ny, nx)
    res = v.view(ny, nx)
    for i, j in pts:
        win = to_host(u0[j - steps:j + steps + 1, i - steps:i + steps + 1]).copy()
        want = oracle.diffuse2d(win, steps, 0.1)[steps, steps]
        got = float(res[j, i])
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (i, j)
    # an edge row of the last step is zero
    assert float(res[ny - 1, 12345]) == 0.0


def test_diffusion_3d_fp32_beyond_2_31_cells():
    torch = torch_cuda()
    from finite_volume_field_gb300 import api
    nx, ny, nz, steps = 1536, 1400, 1000, 2   # 2.15e9 cells
    n = nx * ny * nz
    u = _ramp(torch, n, 999983.0, 0.0, 1e-6, torch.float32)
    v = torch.zeros_like(u)
    api.diffuse3d_step(u, v, nx, ny, nz, 0.1, steps, api.FVF_FP32)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    u0 = _ramp(torch, n, 999983.0, 0.0, 1e-6, torch.float32).view(nz, ny, nx)
    res = u.view(nz, ny, nx)                  # two steps: the result is back in u
    rng = np.random.default_rng(8)
    pts = np.stack([rng.integers(steps, nx - steps, 48), rng.integers(steps, ny - steps, 48),
                    rng.integers(steps, nz - steps, 48)], 1)
    pts = np.concatenate([pts, [[nx - 1 - steps, ny - 1 - steps, nz - 1 - steps]]])
    for i, j, k in pts:
        win = to_host(u0[k - steps:k + steps + 1, j - steps:j + steps + 1,
                         i - steps:i + steps + 1]).copy()
        want = oracle.diffuse3d(win, steps, 0.1)[steps, steps, steps]
        got = float(res[k, j, i])
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (i, j, k)


@pytest.mark.parametrize("direction", [0, 2])
def test_pack_fp64_beyond_2_31_elements(direction):
    """One field of 1300 x 1300 x 1300 interior cells plus 2 ghost layers
    (2.2e9 stored elements, 17.6 GB): out(a,b,c) = field(mapped (j,k,l)) at
    sampled outputs, as the pack's mapping defines."""
    torch = torch_cuda()
    from finite_volume_field_gb300 import api
    n1 = n2 = n3 = 1300
    g = 2
    N1 = N2 = N3 = n1 + 2 * g
    f = _ramp(torch, N1 * N2 * N3, 2 ** 31 - 1, 0.0, 1.0, torch.float64)  # value = index mod p
    M = oracle.pack_extents((n1, n2, n3), g, direction)
    out = torch.empty(M[0] * M[1] * M[2], dtype=torch.float64, device="cuda")
    api.weno_pack([f], 1, (n1, n2, n3), g, direction, out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    a = rng.integers(0, M[0], 4000)
    b = rng.integers(0, M[1], 4000)
    c = rng.integers(0, M[2], 4000)
    a[:2], b[:2], c[:2] = [0, M[0] - 1], [0, M[1] - 1], [0, M[2] - 1]
    if direction == 0:
        j, k, l = a, b + g, c + g
    else:
        j, k, l = c + g, b + g, a
    src = torch.from_numpy(j + N1 * (k + N2 * l)).cuda()
    dst = torch.from_numpy(a + M[0] * (b + M[1] * c)).cuda()
    assert_bits_equal(to_host(out[dst]), to_host(f[src]), what=f"dir {direction}")


@pytest.mark.parametrize("fp32,direction", [(False, 0), (False, 1), (False, 2), (True, 0),
                                            (True, 2)])
def test_flux_difference_beyond_2_31_elements(fp32, direction):
    """One variable on 1300^3 cells (2.2e9 rhs elements, 17.6 GB per FP64
    array): the flux difference at sampled cells equals the oracle's on the
    one-cell case cut around each (its two faces and its inverse width)."""
    torch = torch_cuda()
    from finite_volume_field_gb300 import api
    n = (1300, 1300, 1300)
    fe = list(n)
    fe[direction] += 1
    tdt, ndt = (torch.float32, np.float32) if fp32 else (torch.float64, np.float64)
    F = _ramp(torch, fe[0] * fe[1] * fe[2], 999983.0, 499991.0, 1e-3, tdt)
    rng = np.random.default_rng(10 + direction)
    w = rng.uniform(0.5, 2.0, n[direction]).astype(ndt)
    rhs = torch.empty(n[0] * n[1] * n[2], dtype=tdt, device="cuda")
    fn = api.advect_rhs_f32 if fp32 else api.advect_rhs
    fn(F, torch.from_numpy(w).cuda(), 1, n, direction, rhs)
    torch.cuda.synchronize()
    pts = np.stack([rng.integers(0, n[0], 300), rng.integers(0, n[1], 300),
                    rng.integers(0, n[2], 300)], 1)
    pts = np.concatenate([pts, [[n[0] - 1, n[1] - 1, n[2] - 1], [0, 0, 0]]])
    step = (1, fe[0], fe[0] * fe[1])[direction]
    lo = pts[:, 0] + fe[0] * (pts[:, 1] + fe[1] * pts[:, 2])
    faces = to_host(torch.stack([F[torch.from_numpy(lo).cuda()],
                                 F[torch.from_numpy(lo + step).cuda()]], 1))
    got = to_host(rhs[torch.from_numpy(pts[:, 0] + n[0] * (pts[:, 1] + n[1] * pts[:, 2])).cuda()])
    ui = np.uint32 if fp32 else np.uint64
    for p, fc, g in zip(pts, faces, got):
        want = oracle.advect_rhs(np.ascontiguousarray(fc), w[p[direction]:p[direction] + 1], 1,
                                 (1, 1, 1), direction)
        assert ndt(g).view(ui) == want[0].view(ui), (p, g, want[0])
