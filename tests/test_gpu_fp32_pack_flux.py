"""GPU parity of the FP32 pack (weno_pack_f32) and the FP32 flux difference
(advect_rhs_f32, advect_rhs_add_f32) against the CPU oracle's binary32 forms,
through the C ABI.  The pack is a 4-byte bit copy; the flux difference is one
binary32 subtraction and one multiplication (and one addition when
accumulating) in the same order on both sides: bit for bit, NaN payloads of
arithmetic results excepted."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, canary_intact, guarded, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

SMALL = [((3, 4, 5), 1), ((5, 4, 1), 2), ((6, 3, 2), 3), ((2, 7, 3), 0), ((33, 31, 35), 3),
         ((70, 3, 40), 2), ((1, 1, 1), 2), ((40, 1, 1), 1), ((1, 37, 1), 2), ((65, 66, 1), 2)]


def _f32_fields(seed, nv, extents, g):
    return [f.astype(np.float32) for f in inputs.normal_fields(seed, nv, extents, g)]


def _gpu_pack(torch, fields, extents, g, direction, offset=0):
    nv = len(fields)
    dev = []
    for f in fields:
        whole = torch.empty(f.size + offset, dtype=torch.float32, device="cuda")
        whole[offset:] = to_dev(f)
        dev.append(whole[offset:])
    M = oracle.pack_extents(extents, g, direction)
    n = M[0] * M[1] * M[2] * nv
    whole, out = guarded(torch, n, torch.float32)
    api.weno_pack_f32(dev, nv, extents, g, direction, out)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "pack wrote past its output"
    return to_host(out)


@pytest.mark.parametrize("extents,g", SMALL)
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3, 8])
def test_pack_f32_small(extents, g, direction, nv):
    torch = torch_cuda()
    fields = _f32_fields(inputs.config_seed(3), nv, extents, g)
    got = _gpu_pack(torch, fields, extents, g, direction, offset=nv % 2)
    assert_bits_equal(got, oracle.weno_pack(fields, extents, g, direction),
                      what=f"pack f32 {extents} g={g} dir={direction} nv={nv}")


def test_pack_f32_special_bits_and_max_nv():
    torch = torch_cuda()
    extents, g = (9, 10, 11), 2
    n = int(np.prod(inputs.stored_extents(extents, g)))
    fields = []
    for i in range(64):
        b = (inputs.random_bits(18, i, n) >> np.uint64(32)).astype(np.uint32)
        b[::7] = 0x7FA0BEEF + i          # NaN payloads
        b[1::11] = 0x80000000            # -0.0
        b[2::13] = 0x00000003            # subnormal
        fields.append(b.view(np.float32))
    for direction in range(3):
        got = _gpu_pack(torch, fields, extents, g, direction)
        assert_bits_equal(got, oracle.weno_pack(fields, extents, g, direction), what=f"dir {direction}")


def _rhs_case(seed, nv, extents, direction):
    flux = inputs.face_fluxes(seed, nv, extents, direction).astype(np.float32)
    w = inputs.inverse_spacing(seed, extents[direction], stream=200 + direction).astype(np.float32)
    return flux, w


@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (1, 6, 2), (7, 1, 3), (33, 35, 37),
                                     (130, 3, 9), (1, 1, 1), (64, 64, 1)])
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 5])
def test_rhs_f32_small(extents, direction, nv):
    torch = torch_cuda()
    flux, w = _rhs_case(inputs.config_seed(4), nv, extents, direction)
    n = int(np.prod(extents)) * nv
    whole, rhs = guarded(torch, n, torch.float32)
    api.advect_rhs_f32(to_dev(flux), to_dev(w), nv, extents, direction, rhs)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n)
    assert_bits_equal(to_host(rhs), oracle.advect_rhs(flux, w, nv, extents, direction))
    base = inputs.normal_f64(15, direction, n).astype(np.float32)
    rhs.copy_(to_dev(base))
    api.advect_rhs_add_f32(to_dev(flux), to_dev(w), nv, extents, direction, rhs)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(rhs), oracle.advect_rhs_add(flux, w, nv, extents, direction, base))


def test_rhs_f32_special_values():
    torch = torch_cuda()
    extents, nv = (37, 6, 5), 3
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-45, -3e-39, 3.4e38, -3.4e38],
                        dtype=np.float32)
    for direction in range(3):
        flux, w = _rhs_case(inputs.config_seed(8), nv, extents, direction)
        flux[::7] = np.resize(specials, flux[::7].size)
        w[::3] = np.resize(np.array([0.0, 1e38, np.inf], dtype=np.float32), w[::3].size)
        rhs = torch.empty(int(np.prod(extents)) * nv, dtype=torch.float32, device="cuda")
        api.advect_rhs_f32(to_dev(flux), to_dev(w), nv, extents, direction, rhs)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(rhs), oracle.advect_rhs(flux, w, nv, extents, direction),
                          nan_payloads=False, what=f"dir {direction}")


def test_pack_and_rhs_f32_full_size():
    """8 FP32 fields of 201^3 + 3 ghost layers packed along x, y, z, and the
    FP32 x + y + z right-hand side of 8 variables on 201^3 cells, every
    element compared with the oracle."""
    torch = torch_cuda()
    extents, g, nv = (201, 201, 201), 3, 8
    fields = _f32_fields(inputs.config_seed(3), nv, extents, g)
    dev = [to_dev(f) for f in fields]
    M = oracle.pack_extents(extents, g, 0)
    out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float32, device="cuda")
    for direction in range(3):
        api.weno_pack_f32(dev, nv, extents, g, direction, out)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(out), oracle.weno_pack(fields, extents, g, direction),
                          what=f"pack 207^3 dir {direction}")
    del dev, out
    rhs = torch.empty(201 ** 3 * nv, dtype=torch.float32, device="cuda")
    want = None
    for direction in range(3):
        flux, w = _rhs_case(inputs.config_seed(4), nv, extents, direction)
        fn = api.advect_rhs_f32 if direction == 0 else api.advect_rhs_add_f32
        fn(to_dev(flux), to_dev(w), nv, extents, direction, rhs)
        torch.cuda.synchronize()
        want = (oracle.advect_rhs(flux, w, nv, extents, 0) if direction == 0
                else oracle.advect_rhs_add(flux, w, nv, extents, direction, want))
        assert_bits_equal(to_host(rhs), want, what=f"rhs 201^3 after dir {direction}")
