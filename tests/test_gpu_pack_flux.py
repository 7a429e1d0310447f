"""GPU parity of weno_pack and advect_rhs against the CPU oracle, through the
C ABI.  The pack is a copy and must match bit for bit (NaN payloads and
signed zeros included); the flux difference is one subtraction and one
multiplication in the same order on both sides and must match bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import (assert_bits_equal, canary_intact, guarded, to_dev, to_host,
                            torch_cuda)

pytestmark = pytest.mark.gpu

SMALL = [((3, 4, 5), 1), ((3, 4, 5), 2), ((5, 4, 1), 2), ((6, 3, 2), 3), ((2, 7, 3), 0),
         ((33, 31, 35), 3), ((70, 3, 40), 2), ((1, 1, 1), 2), ((40, 1, 1), 1), ((1, 37, 1), 2),
         ((65, 66, 1), 2)]


def _gpu_pack(torch, fields, extents, g, direction, out_pad=64):
    nv = len(fields)
    dev = [to_dev(f) for f in fields]
    M = oracle.pack_extents(extents, g, direction)
    n = M[0] * M[1] * M[2] * nv
    whole, out = guarded(torch, n, torch.float64, out_pad)
    api.weno_pack(dev, nv, extents, g, direction, out)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "pack wrote past its output"
    return to_host(out)


def _gpu_rhs(torch, flux, inv_d, nv, extents, direction):
    n = extents[0] * extents[1] * extents[2] * nv
    whole, rhs = guarded(torch, n, torch.float64)
    api.advect_rhs(to_dev(flux), to_dev(inv_d), nv, extents, direction, rhs)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "advect_rhs wrote past its output"
    return to_host(rhs)


@pytest.mark.parametrize("extents,g", SMALL)
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3, 8])
def test_pack_small(extents, g, direction, nv):
    torch = torch_cuda()
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    got = _gpu_pack(torch, fields, extents, g, direction)
    want = oracle.weno_pack(fields, extents, g, direction)
    assert_bits_equal(got, want, what=f"pack {extents} g={g} dir={direction} nv={nv}")


def test_pack_special_bits_and_max_nv():
    """NaN payloads, -0.0, infinities and subnormals copy bit for bit; 64
    variables (the maximum) all land in place."""
    torch = torch_cuda()
    extents, g = (9, 10, 11), 2
    n = int(np.prod(inputs.stored_extents(extents, g)))
    fields = []
    for i in range(64):
        b = inputs.random_bits(17, i, n)
        b[::7] = 0x7FF4DEADBEEF0000 + i
        b[1::11] = 0x8000000000000000
        b[2::13] = 0x0000000000000003
        fields.append(b.view(np.float64))
    for direction in range(3):
        got = _gpu_pack(torch, fields, extents, g, direction)
        want = oracle.weno_pack(fields, extents, g, direction)
        assert_bits_equal(got, want, what=f"dir {direction}")


def test_pack_aliasing_fields_and_errors():
    """The same field may appear several times; an output that overlaps a
    field is refused."""
    torch = torch_cuda()
    extents, g = (8, 9, 10), 1
    f = inputs.normal_fields(5, 1, extents, g)[0]
    got = _gpu_pack(torch, [f, f, f], extents, g, 1)
    assert_bits_equal(got, oracle.weno_pack([f, f, f], extents, g, 1))
    big = torch.zeros(10 * f.size, dtype=torch.float64, device="cuda")
    big[: f.size] = torch.from_numpy(f).cuda()
    with pytest.raises(api.FvfError) as e:
        api.weno_pack([big[: f.size]], 1, extents, g, 0, big[f.size // 2:])
    assert e.value.status == 6
    torch.cuda.synchronize()


@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (1, 6, 2), (7, 1, 3), (33, 35, 37),
                                     (130, 3, 9), (1, 1, 1), (64, 64, 1)])
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3, 8])
def test_rhs_small(extents, direction, nv):
    torch = torch_cuda()
    seed = inputs.config_seed(4)
    flux = inputs.face_fluxes(seed, nv, extents, direction)
    inv_d = inputs.inverse_spacing(seed, extents[direction], stream=200 + direction)
    got = _gpu_rhs(torch, flux, inv_d, nv, extents, direction)
    want = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
    assert_bits_equal(got, want, what=f"rhs {extents} dir={direction} nv={nv}")


def test_rhs_special_values_and_alias():
    """inf/NaN/huge/subnormal fluxes (subtraction overflow, products below
    the normal range), zero, subnormal, huge and infinite spacings, in every
    direction and every variable slot of a load batch (the products of some
    slots run on the integer pipes); and an rhs overlapping the flux is
    refused."""
    torch = torch_cuda()
    extents = (17, 9, 5)
    for nv in (3, 5):
        for direction in range(3):
            flux = inputs.face_fluxes(9, nv, extents, direction)
            flux[::5] = 1.7e308
            flux[1::7] = -1.7e308
            flux[2::11] = np.inf
            flux[3::13] = np.nan
            flux[4::17] = -0.0
            flux[5::19] = 5e-324
            flux[6::23] = -2.2e-308
            inv_d = inputs.inverse_spacing(9, extents[direction])
            inv_d[0] = 5e-324
            inv_d[1] = 1e300
            inv_d[2] = 0.0
            inv_d[3] = np.inf
            inv_d[4] = 1e-310
            got = _gpu_rhs(torch, flux, inv_d, nv, extents, direction)
            want = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
            assert_bits_equal(got, want, nan_payloads=False, what=f"dir {direction} nv {nv}")
    nv = 3
    flux = inputs.face_fluxes(9, nv, extents, 0)
    inv_d = inputs.inverse_spacing(9, 17)
    F = to_dev(flux)
    with pytest.raises(api.FvfError) as e:
        api.advect_rhs(F, to_dev(inv_d), nv, extents, 0, F[: 17 * 9 * 5 * nv])
    assert e.value.status == 6
    torch.cuda.synchronize()


def _tie_faces(seed, nv, extents, direction):
    """Face fluxes whose differences are exact values with a set last
    significand bit (every other face zero), so that their products with a
    spacing of few significand bits (1.5, 0.75, 1.25) land exactly halfway
    between two doubles, or one unit either side: round-to-even territory."""
    fl = inputs.face_fluxes(seed, nv, extents, direction)
    bits = fl.view(np.uint64) | np.uint64(1)                    # odd significands
    bits ^= (inputs.random_bits(seed, 900, fl.size) & np.uint64(2))  # and next-to-last bits
    fl = bits.view(np.float64).copy()
    fe = oracle.flux_extents(extents, direction)
    f4 = fl.reshape(nv, fe[2], fe[1], fe[0])
    idx = [np.arange(m) for m in fe]
    mask = (idx[direction] % 2 == 1)
    if direction == 0:
        f4[:, :, :, mask] = 0.0
    elif direction == 1:
        f4[:, :, mask, :] = 0.0
    else:
        f4[:, mask, :, :] = 0.0
    return f4.reshape(-1)


@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [4, 8])
def test_rhs_products_at_rounding_ties(direction, nv):
    """Spacings 1.5, 0.75 and 1.25 times differences with odd significands:
    the exact products sit on or beside rounding ties, where the integer-pipe
    product's sticky bit and ties-to-even decide the last bit.  Assigning and
    accumulating forms, every variable slot of a load batch."""
    torch = torch_cuda()
    extents = (37, 9, 6)
    flux = _tie_faces(21, nv, extents, direction)
    n_dir = extents[direction]
    inv_d = np.resize(np.array([1.5, 0.75, 1.25, -1.5, 3.0 * 2.0 ** -900]), n_dir).astype(np.float64)
    got = _gpu_rhs(torch, flux, inv_d, nv, extents, direction)
    want = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
    assert_bits_equal(got, want, what=f"assign dir {direction}")
    old = inputs.normal_f64(22, direction, got.size)
    rhs = to_dev(old)
    api.advect_rhs_add(to_dev(flux), to_dev(inv_d), nv, extents, direction, rhs)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(rhs), oracle.advect_rhs_add(flux, inv_d, nv, extents, direction, old),
                      what=f"accumulate dir {direction}")


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark uses
# ---------------------------------------------------------------------------

def test_pack_full_size_207_cubed():
    """8 fields of 201^3 interior + 3 ghost layers (207^3 stored), N(0,1):
    packed along x, y and z, every element compared with the oracle."""
    torch = torch_cuda()
    extents, g, nv = (201, 201, 201), 3, 8
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    dev = [to_dev(f) for f in fields]
    M = oracle.pack_extents(extents, g, 0)
    out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float64, device="cuda")
    for direction in range(3):
        api.weno_pack(dev, nv, extents, g, direction, out)
        torch.cuda.synchronize()
        want = oracle.weno_pack(fields, extents, g, direction)
        assert_bits_equal(to_host(out), want, what=f"207^3 dir {direction}")


def test_rhs_full_size_201_cubed():
    """nv = 8, 201^3 cells, face fluxes N(0,1), inv_d = 1/d with
    d ~ U[0.5, 1.5]/201: x, y and z, every element compared."""
    torch = torch_cuda()
    extents, nv = (201, 201, 201), 8
    seed = inputs.config_seed(4)
    rhs = torch.empty(201 ** 3 * nv, dtype=torch.float64, device="cuda")
    for direction in range(3):
        flux = inputs.face_fluxes(seed, nv, extents, direction)
        inv_d = inputs.inverse_spacing(seed, 201, stream=200 + direction)
        api.advect_rhs(to_dev(flux), to_dev(inv_d), nv, extents, direction, rhs)
        torch.cuda.synchronize()
        want = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
        assert_bits_equal(to_host(rhs), want, what=f"201^3 dir {direction}")


def test_multivar_sequence_4800x1200():
    """The 2D multi-variable sequence (7 fields of 4800 x 1200 cells, ghost
    2; pack x, pack y, rhs x, rhs y) repeated 100 times on one stream; every
    output of the last repetition compared with one oracle repetition (each
    pass assigns its output, so repetitions do not accumulate)."""
    torch = torch_cuda()
    extents, g, nv = (4800, 1200, 1), 2, 7
    seed = inputs.config_seed(5)
    fields = inputs.multivar_fields_2d(seed, extents, g)
    fx = inputs.face_fluxes(seed, nv, extents, 0)
    fy = inputs.face_fluxes(seed, nv, extents, 1)
    wx = inputs.inverse_spacing(seed, 4800, stream=200)
    wy = inputs.inverse_spacing(seed, 1200, stream=201)
    df = [to_dev(f) for f in fields]
    dfx, dfy, dwx, dwy = to_dev(fx), to_dev(fy), to_dev(wx), to_dev(wy)
    px = torch.empty(4804 * 1200 * nv, dtype=torch.float64, device="cuda")
    py = torch.empty(1204 * 4800 * nv, dtype=torch.float64, device="cuda")
    rx = torch.empty(4800 * 1200 * nv, dtype=torch.float64, device="cuda")
    ry = torch.empty_like(rx)
    for _ in range(100):
        api.weno_pack(df, nv, extents, g, 0, px)
        api.weno_pack(df, nv, extents, g, 1, py)
        api.advect_rhs(dfx, dwx, nv, extents, 0, rx)
        api.advect_rhs(dfy, dwy, nv, extents, 1, ry)
    torch.cuda.synchronize()
    wpx, wpy, wrx, wry = oracle.multivar_sweep_2d(fields, fx, fy, wx, wy, nv, extents, g)
    assert_bits_equal(to_host(px), wpx, what="pack x")
    assert_bits_equal(to_host(py), wpy, what="pack y")
    assert_bits_equal(to_host(rx), wrx, what="rhs x")
    assert_bits_equal(to_host(ry), wry, what="rhs y")


def test_multivar_sequence_4800x1200_as_cuda_graph():
    """The same sequence in the launch configuration the benchmark times: the
    100 repetitions captured once into a CUDA graph through the same library
    calls, then replayed twice; outputs (cleared before the replays) compared
    with the oracle."""
    torch = torch_cuda()
    extents, g, nv = (4800, 1200, 1), 2, 7
    seed = inputs.config_seed(5)
    fields = inputs.multivar_fields_2d(seed, extents, g)
    fx = inputs.face_fluxes(seed, nv, extents, 0)
    fy = inputs.face_fluxes(seed, nv, extents, 1)
    wx = inputs.inverse_spacing(seed, 4800, stream=200)
    wy = inputs.inverse_spacing(seed, 1200, stream=201)
    df = [to_dev(f) for f in fields]
    dfx, dfy, dwx, dwy = to_dev(fx), to_dev(fy), to_dev(wx), to_dev(wy)
    px = torch.zeros(4804 * 1200 * nv, dtype=torch.float64, device="cuda")
    py = torch.zeros(1204 * 4800 * nv, dtype=torch.float64, device="cuda")
    rx = torch.zeros(4800 * 1200 * nv, dtype=torch.float64, device="cuda")
    ry = torch.zeros_like(rx)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    n0 = api.launch_count()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        s = torch.cuda.current_stream()
        for _ in range(100):
            api.weno_pack(df, nv, extents, g, 0, px, s)
            api.weno_pack(df, nv, extents, g, 1, py, s)
            api.advect_rhs(dfx, dwx, nv, extents, 0, rx, s)
            api.advect_rhs(dfy, dwy, nv, extents, 1, ry, s)
    assert api.launch_count() - n0 == 400
    for t in (px, py, rx, ry):
        t.zero_()
    torch.cuda.synchronize()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    wpx, wpy, wrx, wry = oracle.multivar_sweep_2d(fields, fx, fy, wx, wy, nv, extents, g)
    assert_bits_equal(to_host(px), wpx, what="pack x")
    assert_bits_equal(to_host(py), wpy, what="pack y")
    assert_bits_equal(to_host(rx), wrx, what="rhs x")
    assert_bits_equal(to_host(ry), wry, what="rhs y")


# ---------------------------------------------------------------------------
# Accumulating flux difference and the directional flux copy (unpack)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (33, 35, 37), (130, 3, 9), (1, 1, 1)])
@pytest.mark.parametrize("direction", [0, 1, 2])
def test_rhs_add_small(extents, direction):
    torch = torch_cuda()
    nv = 5
    seed = inputs.config_seed(4)
    flux = inputs.face_fluxes(seed, nv, extents, direction)
    inv_d = inputs.inverse_spacing(seed, extents[direction], stream=220 + direction)
    old = inputs.normal_f64(seed, 320 + direction, int(np.prod(extents)) * nv)
    n = old.size
    whole, rhs = guarded(torch, n, torch.float64)
    rhs.copy_(torch.from_numpy(old).cuda())
    api.advect_rhs_add(to_dev(flux), to_dev(inv_d), nv, extents, direction, rhs)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n)
    want = oracle.advect_rhs_add(flux, inv_d, nv, extents, direction, old)
    assert_bits_equal(to_host(rhs), want, what=f"rhs_add {extents} dir {direction}")


def test_rhs_add_special_values():
    torch = torch_cuda()
    extents, nv = (17, 9, 5), 3
    flux = inputs.face_fluxes(19, nv, extents, 1)
    flux[::5] = 1.7e308
    flux[2::11] = np.inf
    flux[3::13] = np.nan
    inv_d = inputs.inverse_spacing(19, 9)
    old = inputs.normal_f64(19, 7, 17 * 9 * 5 * nv)
    old[::7] = -0.0
    old[1::9] = np.inf
    rhs = to_dev(old)
    api.advect_rhs_add(to_dev(flux), to_dev(inv_d), nv, extents, 1, rhs)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(rhs), oracle.advect_rhs_add(flux, inv_d, nv, extents, 1, old),
                      nan_payloads=False)


@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (1, 6, 2), (33, 31, 35), (70, 3, 40),
                                     (1, 1, 1)])
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 7])
def test_flux_unpack_small(extents, direction, nv):
    torch = torch_cuda()
    size = int(np.prod(oracle.sweep_flux_extents(extents, direction))) * nv
    src = inputs.random_bits(23, direction, size).view(np.float64)   # any bit pattern
    whole, out = guarded(torch, size, torch.float64)
    api.flux_unpack(to_dev(src), nv, extents, direction, out)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, size)
    assert_bits_equal(to_host(out), oracle.flux_unpack(src, nv, extents, direction),
                      what=f"unpack {extents} dir {direction} nv {nv}")


def test_true_fv_rhs_three_directions_full_size():
    """The finite-volume right-hand side on 8 x 201^3: the x term assigned,
    the y and z terms accumulated, each direction's physical-frame fluxes
    first produced from sweep-frame fluxes by the unpack -- every element
    compared with the oracle doing the same."""
    torch = torch_cuda()
    extents, nv = (201, 201, 201), 8
    seed = inputs.config_seed(4)
    rhs = torch.empty(201 ** 3 * nv, dtype=torch.float64, device="cuda")
    want = None
    for direction in range(3):
        sweep = inputs.normal_f64(seed, 400 + direction,
                                  int(np.prod(oracle.sweep_flux_extents(extents, direction))) * nv)
        inv_d = inputs.inverse_spacing(seed, 201, stream=230 + direction)
        phys = torch.empty(sweep.size, dtype=torch.float64, device="cuda")
        api.flux_unpack(to_dev(sweep), nv, extents, direction, phys)
        if direction == 0:
            api.advect_rhs(phys, to_dev(inv_d), nv, extents, 0, rhs)
        else:
            api.advect_rhs_add(phys, to_dev(inv_d), nv, extents, direction, rhs)
        torch.cuda.synchronize()
        pf = oracle.flux_unpack(sweep, nv, extents, direction)
        assert_bits_equal(to_host(phys), pf, what=f"unpack dir {direction}")
        want = (oracle.advect_rhs(pf, inv_d, nv, extents, 0) if direction == 0
                else oracle.advect_rhs_add(pf, inv_d, nv, extents, direction, want))
        del phys
    assert_bits_equal(to_host(rhs), want, what="x + y + z")
