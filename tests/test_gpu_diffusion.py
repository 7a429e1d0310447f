"""GPU parity of diffuse2d_step against the CPU oracle, through the C ABI.

The bar is bit-exactness: the kernel and the oracle evaluate
c + alpha*((((W+E)+S)+N) - 4c) with every operation rounded to nearest even,
so every cell must match bit for bit (NaN payloads excepted).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import (assert_bits_equal, canary_intact, guarded, to_dev, to_host,
                            torch_cuda)

pytestmark = pytest.mark.gpu

DT = {np.float32: api.FVF_FP32, np.float64: api.FVF_FP64}


def _run_gpu(torch, u0: np.ndarray, nsteps: int, alpha=0.1, v0=None, stream=None):
    ny, nx = u0.shape
    u = to_dev(u0)
    v = to_dev(np.zeros_like(u0) if v0 is None else v0)
    api.diffuse2d_step(u, v, nx, ny, alpha, nsteps, DT[u0.dtype.type], stream=stream)
    torch.cuda.synchronize()
    return to_host(u), to_host(v)


@pytest.mark.parametrize("dt", [np.float64, np.float32])
def test_centre_impulse_64x64_32_steps(dt):
    """The 64x64 centre-impulse case, 32 steps (result in u)."""
    torch = torch_cuda()
    u0 = oracle.centre_impulse(64, 64, dt)
    gu, gv = _run_gpu(torch, u0, 32)
    ou, ov, in_v = oracle.diffuse2d(u0, 32, return_both=True)
    assert not in_v
    assert_bits_equal(gu, ou, what="u (result)")
    assert_bits_equal(gv, ov, what="v (previous step)")
    one_u, one_v = _run_gpu(torch, u0, 1)
    assert one_v[31, 31] == dt(0.6) and one_v[31, 32] == dt(0.1)


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("steps", [7, 8, 31, 32])
def test_validation_matrix_31x27(dt, steps):
    """The Qiita page's check matrix (section 10 check scripts): both
    precisions, steps 7/8/31/32 on 31x27; both buffers bit-exact."""
    torch = torch_cuda()
    u0 = oracle.centre_impulse(31, 27, dt)
    gu, gv = _run_gpu(torch, u0, steps)
    ou, ov, in_v = oracle.diffuse2d(u0, steps, return_both=True)
    assert in_v == (steps % 2 == 1)
    assert_bits_equal(gu, ou, what="u")
    assert_bits_equal(gv, ov, what="v")
    res = gv if in_v else gu
    assert oracle.physical_check(res)["ok"]


RAGGED = [(1, 1), (2, 2), (3, 3), (1, 9), (9, 1), (5, 5), (3, 17), (17, 3), (33, 65), (65, 33),
          (127, 129), (130, 7), (1000, 3), (3, 1000), (257, 255), (513, 67)]


@pytest.mark.parametrize("dt", [np.float64, np.float32])
@pytest.mark.parametrize("nx,ny", RAGGED)
def test_ragged_random_fields(dt, nx, ny):
    """Sizes that are not multiples of any block or vector width, tiny
    degenerate grids (no interior) and random values everywhere, edges
    included (the kernel must read source edges as they are and write zero
    edges)."""
    torch = torch_cuda()
    n = nx * ny
    vals = (inputs.uniform_f32(7, nx * 1000 + ny, n) if dt == np.float32
            else inputs.uniform_f64(7, nx * 1000 + ny, n))
    u0 = vals.reshape(ny, nx)
    v0 = (inputs.uniform_f32(8, nx, n) if dt == np.float32
          else inputs.uniform_f64(8, nx, n)).reshape(ny, nx)
    for steps in (1, 2, 5):
        gu, gv = _run_gpu(torch, u0, steps, v0=v0)
        ou, ov, _ = oracle.diffuse2d(u0, steps, v0=v0, return_both=True)
        assert_bits_equal(gu, ou, what=f"u {nx}x{ny} {steps}")
        assert_bits_equal(gv, ov, what=f"v {nx}x{ny} {steps}")


@pytest.mark.parametrize("dt", [np.float64, np.float32])
def test_special_values(dt):
    """Huge values (4c overflows: the kernel's two-operation branch), inf,
    NaN, signed zeros and subnormals, with alpha 0.1, 0.3, 0 and the smallest
    subnormal; bit-exact up to NaN payloads."""
    torch = torch_cuda()
    nx, ny = 37, 23
    rng_bits = inputs.random_bits(3, 1, nx * ny)
    if dt == np.float64:
        u0 = (inputs.uniform_f64(3, 2, nx * ny) - 0.5).reshape(ny, nx)
        specials = [np.inf, -np.inf, np.nan, -0.0, 5e-324, 2.0 ** 1022, -2.0 ** 1023,
                    1.7e308, 2.0 ** -1022, 3.0 * 2.0 ** 1021]
    else:
        u0 = (inputs.uniform_f32(3, 2, nx * ny) - np.float32(0.5)).reshape(ny, nx)
        specials = [np.inf, -np.inf, np.nan, -0.0, 1e-45, 2.0 ** 126, -2.0 ** 127, 3.3e38,
                    2.0 ** -126, 3.0 * 2.0 ** 125]
    flat = u0.reshape(-1)
    for s, b in zip(specials, rng_bits[: len(specials)]):
        flat[int(b % (nx * ny))] = dt(s)
    tiny = 1e-45 if dt == np.float32 else 5e-324
    for alpha in (0.1, 0.3, 0.0, tiny):
        for steps in (1, 3):
            gu, gv = _run_gpu(torch, u0, steps, alpha=alpha)
            ou, ov, _ = oracle.diffuse2d(u0, steps, alpha=alpha, return_both=True)
            assert_bits_equal(gu, ou, nan_payloads=False, what=f"u a={alpha} s={steps}")
            assert_bits_equal(gv, ov, nan_payloads=False, what=f"v a={alpha} s={steps}")


def test_guard_band_and_nonzero_stream():
    """Writes stay inside the nx*ny cells (canaries after both buffers are
    untouched) and the work runs on the caller's stream."""
    torch = torch_cuda()
    nx, ny = 301, 77
    u0 = inputs.diffusion_field(nx, ny, np.float64, seed=inputs.config_seed(2))
    uw, u = guarded(torch, nx * ny, torch.float64)
    vw, v = guarded(torch, nx * ny, torch.float64)
    u.copy_(torch.from_numpy(u0.reshape(-1)))
    v.zero_()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.diffuse2d_step(u, v, nx, ny, 0.1, 9, api.FVF_FP64, stream=s)
    s.synchronize()
    assert canary_intact(torch, uw, nx * ny) and canary_intact(torch, vw, nx * ny)
    want = oracle.diffuse2d(u0, 9)
    assert_bits_equal(to_host(v).reshape(ny, nx), want)


def test_device_errors_are_status_codes():
    """A too-small device buffer or a host pointer is refused before launch."""
    torch = torch_cuda()
    u = torch.zeros(100, dtype=torch.float64, device="cuda")
    v = torch.zeros(100, dtype=torch.float64, device="cuda")
    # 20x20 cells do not fit in 100 elements of a fresh allocation; torch's
    # caching allocator may hand out a larger block, so use a 1 GiB grid.
    with pytest.raises(api.FvfError) as e:
        api.diffuse2d_step(u, v, 1 << 15, 1 << 15, 0.1, 1, api.FVF_FP64)
    assert e.value.status == 10
    h = np.zeros(100)
    with pytest.raises(api.FvfError) as e:
        api.diffuse2d_step(h.ctypes.data, v, 10, 10, 0.1, 1, api.FVF_FP64)
    assert e.value.status == 9
    torch.cuda.synchronize()


def test_launch_count():
    """One kernel launch per step (counted by the library)."""
    torch = torch_cuda()
    u = torch.zeros(64 * 64, dtype=torch.float64, device="cuda")
    v = torch.zeros_like(u)
    before = api.launch_count()
    api.diffuse2d_step(u, v, 64, 64, 0.1, 5, api.FVF_FP64)
    torch.cuda.synchronize()
    assert api.launch_count() - before >= 1


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_full_size_8192_200_steps(dt):
    """The 8192 x 8192, 200-step workload (interior uniform [0,1) from the
    seed, zero edges) in the same launch configuration the benchmark times,
    compared cell by cell with the multithreaded oracle."""
    torch = torch_cuda()
    nx = ny = 8192
    u0 = inputs.diffusion_field(nx, ny, dt, seed=inputs.config_seed(2),
                                stream=0 if dt == np.float32 else 1)
    u = to_dev(u0)
    v = torch.zeros_like(u)
    api.diffuse2d_step(u, v, nx, ny, 0.1, 200, DT[dt])
    torch.cuda.synchronize()
    got = to_host(u)
    del u, v
    want = oracle.diffuse2d(u0, 200, nthreads=oracle.max_threads())
    assert_bits_equal(got, want, what=f"8192^2 {dt.__name__}")
    assert oracle.physical_check(got)["min"] >= 0


@pytest.mark.parametrize("nx,ny", [(512, 256), (1130, 65), (258, 300), (4000, 11)])
def test_mixed_sign_fields(nx, ny):
    """FP64 fields of mixed signs on grids the row-marching kernel takes
    (above 32K cells, rows 16-byte aligned): N(0,1) values in the upper rows,
    their magnitudes in the lower rows (rows of a warp then take either form
    of the integer-pipe additions), a block of zeros and a band of negative
    magnitudes; several step counts, both buffers bit-exact."""
    torch = torch_cuda()
    n = nx * ny
    u0 = inputs.normal_f64(21, nx + ny, n).reshape(ny, nx)
    u0[ny // 2:, :] = np.abs(u0[ny // 2:, :])
    u0[ny // 4: ny // 4 + 9, nx // 3: nx // 3 + 40] = 0.0
    u0[3 * ny // 4: 3 * ny // 4 + 3, :] *= -1.0
    for steps in (1, 2, 5):
        gu, gv = _run_gpu(torch, u0, steps)
        ou, ov, _ = oracle.diffuse2d(u0, steps, return_both=True)
        assert_bits_equal(gu, ou, what=f"u {nx}x{ny} {steps}")
        assert_bits_equal(gv, ov, what=f"v {nx}x{ny} {steps}")


def _binade_field(nx, ny, seed):
    """FP64 field in bands of 8 rows, each band built from sign, exponent and
    fraction bits so that the four neighbours of a cell meet one boundary of
    the march kernel's fixed-point neighbour sum: exponents spread over at
    most 9 binades (accepted) or 10 (declined), significands of at most four
    bits (rounding ties in the partial sums), all-ones significands, largest
    exponents on both sides of the 2^1020 bound (sums that overflow
    included) and of the 2^-1013 bound, zeros and subnormals, negative bands,
    and rows of mixed signs."""
    n = nx * ny
    b = inputs.random_bits(seed, 1, 3 * n).reshape(3, ny, nx)
    frac = b[0] & np.uint64((1 << 52) - 1)
    u8 = (b[1] & np.uint64(0xFF)).astype(np.int64)
    mode = (np.arange(ny) // 8) % 10
    u0 = np.zeros((ny, nx), dtype=np.float64)
    for m in range(10):
        rows = mode == m
        fr, r = frac[rows], u8[rows]
        if m == 0:       # spread <= 9 binades about 2^0
            e = 1023 - r % 10
        elif m == 1:     # spread up to 10 binades
            e = 1023 - r % 11
        elif m == 2:     # four-bit significands, spread 3: ties
            e = 1023 - r % 4
            fr = fr & np.uint64(0xF << 48)
        elif m == 3:     # all-ones significands, spread 9
            e = 1023 - r % 10
            fr = np.full_like(fr, (1 << 52) - 1)
        elif m == 4:     # largest exponents about 2^1020: both sides of the range bound
            e = 2045 - r % 6
        elif m == 5:     # largest exponents about 2^-1013: both sides of the lower bound
            e = 12 - r % 6
        elif m == 6:     # zeros and subnormals among normal values
            e = np.where(r % 5 == 0, 0, 1023 - r % 4)
            fr = np.where(r % 10 == 0, np.uint64(0), fr)
        elif m == 7:     # negative band, spread <= 9
            e = 1023 - r % 10
        elif m == 8:     # mixed signs in every row
            e = 1023 - r % 3
        else:            # spread exactly 9 and 10 in alternating columns
            e = np.where((np.arange(nx)[None, :] % 2) == 0, 1023, 1014 - (r % 2))
            e = np.broadcast_to(e, fr.shape)
        sign = np.uint64(1 << 63) if m == 7 else (
            ((b[2][rows] & np.uint64(1)) << np.uint64(63)) if m == 8 else np.uint64(0))
        bits = sign | (np.asarray(e, dtype=np.uint64) << np.uint64(52)) | fr
        u0[rows] = bits.view(np.float64)
    u0[0, :] = u0[-1, :] = 0.0
    u0[:, 0] = u0[:, -1] = 0.0
    return u0


@pytest.mark.parametrize("nx,ny", [(1024, 160), (2050, 88)])
def test_fixed_point_sum_boundaries(nx, ny):
    """FP64 on grids the march kernel takes: every boundary of the
    fixed-point neighbour sum (spread, range, ties, zeros, subnormals, signs),
    1 and 2 steps, both buffers bit-exact up to NaN payloads (the bands near
    2^1021 overflow to infinities and NaNs)."""
    torch = torch_cuda()
    u0 = _binade_field(nx, ny, 31)
    for steps in (1, 2):
        gu, gv = _run_gpu(torch, u0, steps)
        ou, ov, _ = oracle.diffuse2d(u0, steps, return_both=True)
        assert_bits_equal(gu, ou, nan_payloads=False, what=f"u {nx}x{ny} {steps}")
        assert_bits_equal(gv, ov, nan_payloads=False, what=f"v {nx}x{ny} {steps}")


def _zero_slot_field(nx, ny, seed, sh=9):
    """FP64 field in bands of 4 rows for the zero-tolerant neighbour sum of
    the cells next to the x edges: positive rows with +0 edges, negative rows
    with +0 edges, positive rows with -0 edges, rows whose columns 2 and
    nx-3 (the zero's partner in the sum of columns 1 and nx-2) lie sh-1, sh
    and sh+1 binades below their neighbours (the form must take the first
    and decline the others), rows with +0 and -0 scattered inside, the same
    with mixed signs, and rows with nonzero edge values."""
    b = inputs.random_bits(seed, 5, 3 * nx * ny).reshape(3, ny, nx)
    u0 = 0.5 + (b[0] >> np.uint64(11)).astype(np.float64) * 2.0 ** -54    # [0.5, 1)
    mode = (np.arange(ny) // 4) % 7
    zeros = (b[1] % np.uint64(7)) == 0
    neg = (b[2] & np.uint64(1)).astype(bool)
    for j in range(ny):
        m = mode[j]
        if m == 1:
            u0[j] = -u0[j]
        elif m == 3:
            k = (sh - 1) + j % 3
            u0[j, 2] *= 2.0 ** -k
            u0[j, nx - 3] *= 2.0 ** -k
        elif m in (4, 5):
            if m == 5:
                u0[j, neg[j]] = -u0[j, neg[j]]
            z = zeros[j]
            u0[j, z] = np.where(neg[j, z], -0.0, 0.0)
    edge = np.where(mode == 2, -0.0, 0.0)
    keep = mode == 6
    u0[~keep, 0] = edge[~keep]
    u0[~keep, nx - 1] = edge[~keep]
    u0[0, :] = u0[-1, :] = 0.0
    return u0


@pytest.mark.parametrize("nx,ny", [(1024, 60), (1030, 33), (258, 140)])
def test_zero_neighbour_slots(nx, ny):
    """FP64 march kernel on fields that exercise the zero-tolerant neighbour
    sum of the column blocks holding an x edge and the edge cells that skip
    the fallback: +0 and -0 edges, negative fields, zero partners' binade
    limit, scattered zeros of both signs; 1 and 2 steps, both buffers
    bit-exact."""
    torch = torch_cuda()
    u0 = _zero_slot_field(nx, ny, 61)
    for steps in (1, 2):
        gu, gv = _run_gpu(torch, u0, steps)
        ou, ov, _ = oracle.diffuse2d(u0, steps, return_both=True)
        assert_bits_equal(gu, ou, what=f"u {nx}x{ny} {steps}")
        assert_bits_equal(gv, ov, what=f"v {nx}x{ny} {steps}")


@pytest.mark.parametrize("alpha", [0.25, 1.0 / 3.0, 0.0, 1e-300, 0.1 + 2.0 ** -50])
def test_march_alpha_values(alpha):
    """FP64 march kernel (1024 x 48, above the cluster kernel's size) with
    alpha at the stability limit, above it, zero, tiny (products deep in the
    subnormal range) and 0.1 plus one unit in its last place; a mixed-sign
    field, 1 and 3 steps, both buffers bit-exact."""
    torch = torch_cuda()
    nx, ny = 1024, 48
    u0 = inputs.normal_f64(33, 4, nx * ny).reshape(ny, nx)
    u0[ny // 2:, :] = np.abs(u0[ny // 2:, :])
    for steps in (1, 3):
        gu, gv = _run_gpu(torch, u0, steps, alpha=alpha)
        ou, ov, _ = oracle.diffuse2d(u0, steps, alpha=alpha, return_both=True)
        assert_bits_equal(gu, ou, what=f"u alpha={alpha} {steps}")
        assert_bits_equal(gv, ov, what=f"v alpha={alpha} {steps}")


def test_full_size_normal_field():
    """The 8192 x 8192 FP64 grid with interior N(0,1) values (mixed signs),
    20 steps, in the launch configuration the benchmark times, cell by cell
    against the multithreaded oracle."""
    torch = torch_cuda()
    nx = ny = 8192
    u0 = inputs.diffusion_field(nx, ny, np.float64, seed=inputs.config_seed(2), stream=2,
                                values="normal")
    u = to_dev(u0)
    v = torch.zeros_like(u)
    api.diffuse2d_step(u, v, nx, ny, 0.1, 20, api.FVF_FP64)
    torch.cuda.synchronize()
    got = to_host(u)
    del u, v
    want = oracle.diffuse2d(u0, 20, nthreads=oracle.max_threads())
    assert_bits_equal(got, want, what="8192^2 N(0,1) FP64")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
@pytest.mark.parametrize("nx,ny", [(300, 250), (1130, 65), (224, 160), (4000, 11), (9, 6000),
                                   (113, 65), (224, 128), (1000, 7), (9, 600)])
@pytest.mark.parametrize("steps", [3, 4, 9, 16, 17, 24])
def test_blocked_steps_multi_tile(dt, nx, ny, steps):
    """Step counts that take the shared-memory blocked path in FP32 (up to 8
    steps per launch, the last step on its own) on grids above the cluster
    kernel's 32K cells, and the 16- or 8-block cluster kernel on smaller
    ones; FP64 takes one launch per step above 32K cells.  Several tiles,
    ragged tile edges, random values everywhere including the edges; both
    buffers bit-exact (the other buffer must hold step n-1)."""
    torch = torch_cuda()
    n = nx * ny
    u0 = (inputs.uniform_f32(11, nx + ny, n) if dt == np.float32
          else inputs.uniform_f64(11, nx + ny, n)).reshape(ny, nx)
    gu, gv = _run_gpu(torch, u0, steps)
    ou, ov, _ = oracle.diffuse2d(u0, steps, return_both=True)
    assert_bits_equal(gu, ou, what=f"u {nx}x{ny} {steps}")
    assert_bits_equal(gv, ov, what=f"v {nx}x{ny} {steps}")
