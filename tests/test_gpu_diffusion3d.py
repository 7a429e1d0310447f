"""GPU parity of diffuse3d_step (3D 7-point diffusion, FP32 and FP64) against
the CPU oracle, through the C ABI.  Both sides evaluate
c + alpha*((((((W+E)+S)+N)+B)+T) - 6c) with every operation rounded to
nearest even, so every cell of both buffers must match bit for bit (NaN
payloads excepted)."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, canary_intact, guarded, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

DT = {np.float32: api.FVF_FP32, np.float64: api.FVF_FP64}
# (nz, ny, nx): 16-byte rows (vector path: nx a multiple of 4 FP32 / 2 FP64) and
# ragged rows (one element per lane), several tiles along i (32 lanes x 4 or 2) and
# j (8 rows), several runs of planes along k, and the degenerate sizes.
SHAPES = [(9, 10, 12), (5, 6, 7), (3, 3, 3), (1, 5, 5), (4, 1, 9), (6, 7, 1), (2, 2, 2),
          (20, 17, 130), (11, 33, 129), (40, 9, 64), (17, 12, 257), (12, 25, 66)]


def _field(shape, dt, seed, zero_edges=True):
    u = inputs.uniform_f64(seed, 0, int(np.prod(shape))).reshape(shape).astype(dt)
    if zero_edges:
        u[0], u[-1] = 0, 0
        u[:, 0], u[:, -1] = 0, 0
        u[:, :, 0], u[:, :, -1] = 0, 0
    return u


def _run(torch, u0, steps, alpha=0.1, v0=None):
    nz, ny, nx = u0.shape
    n = u0.size
    tdt = torch.float64 if u0.dtype == np.float64 else torch.float32
    wu, u = guarded(torch, n, tdt)
    wv, v = guarded(torch, n, tdt)
    u.copy_(to_dev(u0.reshape(-1)))
    v.copy_(to_dev((np.zeros_like(u0) if v0 is None else v0).reshape(-1)))
    api.diffuse3d_step(u, v, nx, ny, nz, alpha, steps, DT[u0.dtype.type])
    torch.cuda.synchronize()
    assert canary_intact(torch, wu, n) and canary_intact(torch, wv, n), "wrote past a buffer"
    return to_host(u).reshape(u0.shape), to_host(v).reshape(u0.shape)


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("steps", [1, 2, 5])
def test_small_grids(dt, shape, steps):
    torch = torch_cuda()
    u0 = _field(shape, dt, 31, zero_edges=False)
    v0 = _field(shape, dt, 32, zero_edges=False)   # the first step must overwrite v's edges
    gu, gv = _run(torch, u0, steps, v0=v0)
    ou, ov, _ = oracle.diffuse3d(u0, steps, 0.1, v0=v0, return_both=True)
    assert_bits_equal(gu, ou, what=f"u {shape} {steps}")
    assert_bits_equal(gv, ov, what=f"v {shape} {steps}")


def _binade_field_3d(shape, seed):
    """FP64 3D field in slabs of 4 planes, each built from sign, exponent and
    fraction bits so that a cell's six neighbours meet one boundary of the
    six-operand fixed-point sum: spreads of at most 8 binades (accepted) or 9
    (declined), significands of at most four bits (ties), all-ones
    significands, exponents about 2^1020 and 2^-1014, zeros and subnormals,
    a negative slab and mixed signs."""
    nz, ny, nx = shape
    n = nz * ny * nx
    b = inputs.random_bits(seed, 2, 3 * n).reshape(3, nz, ny, nx)
    frac = b[0] & np.uint64((1 << 52) - 1)
    r = (b[1] & np.uint64(0xFF)).astype(np.int64)
    u0 = np.zeros(shape, dtype=np.float64)
    for k in range(nz):
        m = (k // 4) % 8
        fr, rk = frac[k], r[k]
        e = {0: 1023 - rk % 9, 1: 1023 - rk % 10, 2: 1023 - rk % 3, 3: 1023 - rk % 9,
             4: 2045 - rk % 6, 5: 11 - rk % 6, 6: np.where(rk % 5 == 0, 0, 1023 - rk % 4),
             7: 1023 - rk % 3}[m]
        if m == 2:
            fr = fr & np.uint64(0xF << 48)
        if m == 3:
            fr = np.full_like(fr, (1 << 52) - 1)
        if m == 6:
            fr = np.where(rk % 10 == 0, np.uint64(0), fr)
        sign = np.uint64(1 << 63) if m == 3 else (
            ((b[2][k] & np.uint64(1)) << np.uint64(63)) if m == 7 else np.uint64(0))
        u0[k] = (sign | (np.asarray(e, dtype=np.uint64) << np.uint64(52)) | fr).view(np.float64)
    u0[0], u0[-1] = 0, 0
    u0[:, 0], u0[:, -1] = 0, 0
    u0[:, :, 0], u0[:, :, -1] = 0, 0
    return u0


@pytest.mark.parametrize("shape", [(34, 20, 130), (40, 9, 64)])
def test_fixed_point_sum_boundaries(shape):
    """FP64 march kernel on fields that meet every boundary of the
    six-operand fixed-point sum, 1 and 2 steps, both buffers bit-exact up to
    NaN payloads (the slabs near 2^1021 overflow)."""
    torch = torch_cuda()
    u0 = _binade_field_3d(shape, 41)
    for steps in (1, 2):
        gu, gv = _run(torch, u0, steps)
        ou, ov, _ = oracle.diffuse3d(u0, steps, 0.1, return_both=True)
        assert_bits_equal(gu, ou, nan_payloads=False, what=f"u {shape} {steps}")
        assert_bits_equal(gv, ov, nan_payloads=False, what=f"v {shape} {steps}")


def _zero_slot_field_3d(shape, seed):
    """FP64 3D field in slabs of 2 planes for the zero-tolerant neighbour sum
    of the cells next to the x faces: positive with +0 faces, negative with
    +0 faces, -0 faces, the zero's partner (columns 2 and nx-3) 7, 8 and 9
    binades below the other neighbours (taken, declined, declined), +0 and
    -0 scattered inside, the same with mixed signs, nonzero x-face values."""
    nz, ny, nx = shape
    n = nz * ny * nx
    b = inputs.random_bits(seed, 6, 3 * n).reshape(3, nz, ny, nx)
    u0 = 0.5 + (b[0] >> np.uint64(11)).astype(np.float64) * 2.0 ** -54
    zeros = (b[1] % np.uint64(7)) == 0
    neg = (b[2] & np.uint64(1)).astype(bool)
    for k in range(nz):
        m = (k // 2) % 7
        if m == 1:
            u0[k] = -u0[k]
        elif m == 3:
            for j in range(ny):
                s = 7 + j % 3
                u0[k, j, 2] *= 2.0 ** -s
                u0[k, j, nx - 3] *= 2.0 ** -s
        elif m in (4, 5):
            if m == 5:
                u0[k][neg[k]] = -u0[k][neg[k]]
            z = zeros[k]
            u0[k][z] = np.where(neg[k][z], -0.0, 0.0)
        if m != 6:
            u0[k, :, 0] = u0[k, :, nx - 1] = -0.0 if m == 2 else 0.0
    u0[0], u0[-1] = 0, 0
    u0[:, 0], u0[:, -1] = 0, 0
    return u0


@pytest.mark.parametrize("shape", [(28, 10, 130), (15, 7, 200), (14, 5, 64)])
def test_zero_neighbour_slots(shape):
    """FP64 march kernel on fields that exercise the zero-tolerant W/E slot
    of the six-operand sum and the face cells that skip the fallback: +0 and
    -0 faces, negative fields, the partner's binade limit, scattered zeros
    of both signs; 1 and 2 steps, both buffers bit-exact."""
    torch = torch_cuda()
    u0 = _zero_slot_field_3d(shape, 63)
    for steps in (1, 2):
        gu, gv = _run(torch, u0, steps)
        ou, ov, _ = oracle.diffuse3d(u0, steps, 0.1, return_both=True)
        assert_bits_equal(gu, ou, what=f"u {shape} {steps}")
        assert_bits_equal(gv, ov, what=f"v {shape} {steps}")


@pytest.mark.parametrize("alpha", [1.0 / 6.0, 0.25, 0.0, 1e-300])
def test_fp64_alpha_values(alpha):
    """FP64 register kernel with alpha at the 3D stability limit (1/6),
    above it, zero and tiny, on a field whose upper half is positive (the
    fixed-point sum) and lower half mixed in sign (the FP64 fallback); 1 and 3
    steps, both buffers bit-exact."""
    torch = torch_cuda()
    shape = (20, 18, 66)
    u0 = inputs.normal_f64(34, 5, int(np.prod(shape))).reshape(shape)
    u0[shape[0] // 2:] = np.abs(u0[shape[0] // 2:])
    for steps in (1, 3):
        gu, gv = _run(torch, u0, steps, alpha=alpha)
        ou, ov, _ = oracle.diffuse3d(u0, steps, alpha, return_both=True)
        assert_bits_equal(gu, ou, what=f"u alpha={alpha} {steps}")
        assert_bits_equal(gv, ov, what=f"v alpha={alpha} {steps}")


@pytest.mark.parametrize("dt", [np.float64, np.float32])
def test_impulse_and_special_values(dt):
    """A centre impulse (exact one-step values at alpha = 1/8), then a field
    with infinities, NaNs, signed zeros and subnormals."""
    torch = torch_cuda()
    u0 = np.zeros((9, 10, 12), dtype=dt)
    u0[4, 5, 6] = 1
    _, gv = _run(torch, u0, 1, alpha=0.125)
    assert gv[4, 5, 6] == dt(0.25) and gv[4, 5, 7] == dt(0.125) and gv[3, 5, 6] == dt(0.125)
    u0 = _field((8, 9, 16), dt, 33)
    flat = u0.reshape(-1)
    specials = np.array([np.inf, -np.inf, np.nan, -0.0, 1e-40 if dt == np.float32 else 1e-310,
                         3e38 if dt == np.float32 else 1.7e308], dtype=dt)
    flat[::17] = np.resize(specials, flat[::17].size)
    # alpha 0 and a subnormal alpha: every product takes the complete
    # (slow-path) multiplication; 1/6 and 0.1 the fixed-factor fast path
    tiny = 1e-40 if dt == np.float32 else 5e-324
    for alpha in (0.1, 1.0 / 6.0, 0.0, tiny):
        gu, gv = _run(torch, u0, 3, alpha=alpha)
        ou, ov, _ = oracle.diffuse3d(u0, 3, alpha, return_both=True)
        assert_bits_equal(gu, ou, nan_payloads=False, what=f"u alpha={alpha}")
        assert_bits_equal(gv, ov, nan_payloads=False, what=f"v alpha={alpha}")


def test_misaligned_rows_take_the_scalar_path():
    """Buffers that start 4 bytes into an allocation (FP32) are not 16-byte
    aligned: the same results through the one-element-per-lane kernel."""
    torch = torch_cuda()
    shape = (7, 9, 64)
    u0 = _field(shape, np.float32, 34)
    n = u0.size
    bu = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    bv = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    bu[1:] = to_dev(u0.reshape(-1))
    api.diffuse3d_step(bu[1:], bv[1:], 64, 9, 7, 0.1, 4, api.FVF_FP32)
    torch.cuda.synchronize()
    ou = oracle.diffuse3d(u0, 4, 0.1)
    assert_bits_equal(to_host(bu[1:]).reshape(shape), ou)


def test_launch_count_and_errors():
    torch = torch_cuda()
    u = torch.zeros(6 * 7 * 8, dtype=torch.float64, device="cuda")
    v = torch.zeros_like(u)
    before = api.launch_count()
    api.diffuse3d_step(u, v, 8, 7, 6, 0.1, 5, api.FVF_FP64)
    torch.cuda.synchronize()
    assert api.launch_count() - before == 5
    with pytest.raises(api.FvfError) as e:
        api.diffuse3d_step(u, u[8:], 8, 7, 5, 0.1, 1, api.FVF_FP64)
    assert e.value.status == 6
    # a grid far larger than the 336-element buffers (torch's caching
    # allocator may hand out a larger block than asked for, but not 8 GiB)
    with pytest.raises(api.FvfError) as e:
        api.diffuse3d_step(u, v, 1024, 1024, 1024, 0.1, 1, api.FVF_FP64)
    assert e.value.status == 10


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_full_size_512_cubed_20_steps(dt):
    """512^3, 20 steps, interior uniform [0,1) with zero boundary faces: both
    buffers compared cell by cell with the oracle (run on all host cores)."""
    torch = torch_cuda()
    shape = (512, 512, 512)
    u0 = _field(shape, dt, 35)
    du = to_dev(u0.reshape(-1))
    dv = torch.zeros_like(du)
    api.diffuse3d_step(du, dv, 512, 512, 512, 0.1, 20, DT[dt])
    torch.cuda.synchronize()
    ou, ov, _ = oracle.diffuse3d(u0, 20, 0.1, nthreads=os.cpu_count() or 1, return_both=True)
    assert_bits_equal(to_host(du).reshape(shape), ou, what="512^3 u")
    assert_bits_equal(to_host(dv).reshape(shape), ov, what="512^3 v")


def test_no_expired_waits():
    """The bulk-copy kernel bounds its waits on its own copies and flags an
    expired one on the device; after the runs above and a few more the flag
    is clear."""
    torch = torch_cuda()
    for shape in ((40, 33, 256), (70, 9, 64)):
        for dt in (np.float32, np.float64):
            u0 = _field(shape, dt, 36)
            gu, gv = _run(torch, u0, 3)
            assert_bits_equal(gv, oracle.diffuse3d(u0, 3, 0.1))
    assert api.device_error() == 0
