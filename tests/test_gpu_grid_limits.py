"""GPU parity at the launch-grid limits of the kernels whose grids walk an
axis with blockIdx.y or blockIdx.z, through the C ABI, against the CPU
oracle (bit for bit):

* the x pack and the x pack fused with the conservative-variable copy take
  one grid row per plane, capped at 65535 rows: with more planes every block
  row loops over several planes;
* the FP64 2D march kernel takes bands of 12 rows: when ny / 12 would exceed
  the 65535 grid rows the bands grow;
* the FP64 3D kernel takes runs of 16 planes: when nz / 16 would exceed the
  65535 grid slices the runs grow.
Each case is small in memory (at most about 140 MB) and long along the
walked axis."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import (assert_bits_equal, canary_intact, guarded, to_dev, to_host,
                            torch_cuda)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp32", [False, True])
def test_pack_x_more_planes_than_grid_rows(fp32):
    torch = torch_cuda()
    extents, g, nv = (3, 2, 70001), 1, 2
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    if fp32:
        fields = [f.astype(np.float32) for f in fields]
    tdt = torch.float32 if fp32 else torch.float64
    n = (extents[0] + 2 * g) * extents[1] * extents[2] * nv   # N1 * n2 * n3 * nv
    whole, out = guarded(torch, n, tdt)
    dev = [torch.from_numpy(np.ascontiguousarray(f)).to("cuda") for f in fields]
    (api.weno_pack_f32 if fp32 else api.weno_pack)(dev, nv, extents, g, 0, out)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "pack wrote past its output"
    want = oracle.weno_pack(fields, extents, g, 0)   # FP32 fields: the 4-byte form
    assert_bits_equal(to_host(out), want, what=f"pack x fp32={fp32}")


def test_pack_copy_x_more_planes_than_grid_rows():
    torch = torch_cuda()
    extents, g, nv = (3, 2, 70001), 1, 2
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    stored = fields[0].size
    n = (extents[0] + 2 * g) * extents[1] * extents[2] * nv
    whole, out = guarded(torch, n, torch.float64)
    copies = [guarded(torch, stored, torch.float64) for _ in range(nv)]
    dev = [to_dev(f) for f in fields]
    api.weno_pack_copy(dev, nv, extents, g, 0, out, [c[1] for c in copies])
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "pack wrote past its output"
    want_pack, want_copies = oracle.weno_pack_copy(fields, extents, g, 0)
    assert_bits_equal(to_host(out), want_pack, what="pack x (fused)")
    for (w, c), f in zip(copies, want_copies):
        assert canary_intact(torch, w, stored), "copy wrote past its output"
        assert_bits_equal(to_host(c), f, what="copy (fused)")


def test_diffusion_fp64_bands_beyond_grid_rows():
    """16 x 1600020: ny / 24 > 65535, so the bands take 25 rows."""
    torch = torch_cuda()
    nx, ny = 16, 1600020
    u0 = inputs.diffusion_field(nx, ny, np.float64, seed=inputs.config_seed(2), stream=7)
    for steps in (1, 2):
        u = to_dev(u0)
        v = torch.zeros_like(u)
        api.diffuse2d_step(u, v, nx, ny, 0.1, steps, api.FVF_FP64)
        torch.cuda.synchronize()
        ou, ov, _ = oracle.diffuse2d(u0, steps, return_both=True)
        assert_bits_equal(to_host(u).reshape(ny, nx), ou, what=f"u {nx}x{ny} {steps} steps")
        assert_bits_equal(to_host(v).reshape(ny, nx), ov, what=f"v {nx}x{ny} {steps} steps")
        del u, v


def test_diffusion3d_fp64_runs_beyond_grid_slices():
    """4 x 4 x 1048600: nz / 16 > 65535, so the runs take 17 planes."""
    torch = torch_cuda()
    shape = (1048600, 4, 4)
    u0 = inputs.uniform_f64(inputs.config_seed(4), 9, int(np.prod(shape))).reshape(shape)
    for steps in (1, 2):
        u = to_dev(u0.reshape(-1))
        v = torch.zeros_like(u)
        api.diffuse3d_step(u, v, 4, 4, shape[0], 0.1, steps, api.FVF_FP64)
        torch.cuda.synchronize()
        ou, ov, _ = oracle.diffuse3d(u0, steps, 0.1, return_both=True)
        assert_bits_equal(to_host(u).reshape(shape), ou, what=f"u 3D {shape} {steps} steps")
        assert_bits_equal(to_host(v).reshape(shape), ov, what=f"v 3D {shape} {steps} steps")
        del u, v
