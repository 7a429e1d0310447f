"""GPU parity of ssprk3_axpby and ssprk3_stage (the SSPRK3 stage update,
alone and fused with the flux difference) against the CPU oracle, through the
C ABI.  Every operation is rounded to nearest even in the same order on both
sides, so results must match bit for bit; NaN results match any NaN (the
payload of an arithmetic NaN is not part of the contract)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, canary_intact, guarded, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

# Shu-Osher SSPRK3 stage coefficients (a, b) and one off-table pair.
COEFS = [(0.0, 1.0), (0.75, 0.25), (1.0 / 3.0, 2.0 / 3.0), (-1.25, 3.5)]
SHAPES = [(3, 4, 5), (1, 1, 1), (7, 1, 1), (1, 9, 1), (1, 1, 6), (33, 31, 35), (65, 66, 1),
          (257, 3, 2), (16, 16, 16), (130, 5, 9)]


def _case(seed, extents, nv):
    n = int(np.prod(extents)) * nv
    fl = [inputs.face_fluxes(seed, nv, extents, d) for d in range(3)]
    w = [inputs.inverse_spacing(seed, extents[d], stream=200 + d) for d in range(3)]
    u0 = inputs.normal_f64(seed, 300, n)
    u = inputs.normal_f64(seed, 301, n)
    return fl, w, u0, u


def _gpu_stage(torch, u0, u, fl, w, nv, extents, a, b, dt):
    n = u.size
    whole, out = guarded(torch, n, torch.float64)
    api.ssprk3_stage(to_dev(u0), to_dev(u), [to_dev(f) if f is not None else None for f in fl],
                     [to_dev(x) for x in w], nv, extents, a, b, dt, out)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole, n), "ssprk3_stage wrote past its output"
    return to_host(out)


@pytest.mark.parametrize("extents", SHAPES)
@pytest.mark.parametrize("nv", [1, 3, 8])
def test_axpby_small(extents, nv):
    torch = torch_cuda()
    seed = inputs.config_seed(6)
    _, _, u0, u = _case(seed, extents, nv)
    rhs = inputs.normal_f64(seed, 302, u.size)
    for a, b in COEFS:
        whole, out = guarded(torch, u.size, torch.float64)
        api.ssprk3_axpby(to_dev(u0), to_dev(u), to_dev(rhs), nv, extents, a, b, 0.37, out)
        torch.cuda.synchronize()
        assert canary_intact(torch, whole, u.size)
        assert_bits_equal(to_host(out), oracle.rk_axpby(u0, u, rhs, a, b, 0.37),
                          what=f"axpby {extents} nv={nv} a={a}")


@pytest.mark.parametrize("extents", SHAPES)
@pytest.mark.parametrize("present", [(0,), (0, 1), (0, 2), (0, 1, 2)])
@pytest.mark.parametrize("nv", [1, 5])
def test_stage_small(extents, present, nv):
    torch = torch_cuda()
    fl, w, u0, u = _case(inputs.config_seed(7), extents, nv)
    f = [fl[d] if d in present else None for d in range(3)]
    for a, b in COEFS:
        got = _gpu_stage(torch, u0, u, f, w, nv, extents, a, b, 0.21)
        want = oracle.ssprk3_stage(u0, u, f, w, nv, extents, a, b, 0.21)
        assert_bits_equal(got, want, what=f"stage {extents} {present} nv={nv} a={a}")


def test_special_values():
    """Infinities, NaNs, signed zeros, subnormals and overflow in every
    input, the inverse spacings included; zero and subnormal coefficients (the
    integer-pipe products then take their complete path); a = 0 still
    multiplies u0 (0*inf = NaN)."""
    torch = torch_cuda()
    extents, nv = (37, 6, 5), 2
    fl, w, u0, u = _case(inputs.config_seed(8), extents, nv)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 5e-324, -2.5e-320, 1.7e308,
                         -1.7e308, 1e-310], dtype=np.float64)
    for arr, step in ((u0, 7), (u, 11), (fl[0], 13), (fl[1], 17), (fl[2], 19)):
        arr[::step] = np.resize(specials, arr[::step].size)
    rhs = inputs.normal_f64(9, 0, u.size)
    rhs[::5] = np.resize(specials, rhs[::5].size)
    for d, x in enumerate(w):
        x[d::4] = np.resize(np.array([0.0, 5e-324, 1e300, np.inf]), x[d::4].size)
    for a, b in COEFS + [(0.0, 0.0), (5e-324, -1e-310)]:
        for dt in (1e300, 0.21, 0.0, 5e-324):
            got = _gpu_stage(torch, u0, u, fl, w, nv, extents, a, b, dt)
            assert_bits_equal(got, oracle.ssprk3_stage(u0, u, fl, w, nv, extents, a, b, dt),
                              nan_payloads=False, what=f"special stage a={a} dt={dt}")
        out = torch.empty(u.size, dtype=torch.float64, device="cuda")
        api.ssprk3_axpby(to_dev(u0), to_dev(u), to_dev(rhs), nv, extents, a, b, 0.5, out)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(out), oracle.rk_axpby(u0, u, rhs, a, b, 0.5),
                          nan_payloads=False, what=f"special axpby a={a}")


def test_in_place_stages_and_alias_rules():
    """out may be u or u0 itself (the stage written in place); a partial
    overlap with them, or any overlap with a flux or an inverse width, is
    refused with nothing launched."""
    torch = torch_cuda()
    extents, nv = (40, 9, 7), 4
    fl, w, u0, u = _case(inputs.config_seed(10), extents, nv)
    dfl = [to_dev(f) for f in fl]
    dw = [to_dev(x) for x in w]
    a, b, dt = 0.75, 0.25, 0.3
    want = oracle.ssprk3_stage(u0, u, fl, w, nv, extents, a, b, dt)
    du0, du = to_dev(u0), to_dev(u)
    api.ssprk3_stage(du0, du, dfl, dw, nv, extents, a, b, dt, du)       # out is u
    torch.cuda.synchronize()
    assert_bits_equal(to_host(du), want, what="in place into u")
    du0, du = to_dev(u0), to_dev(u)
    api.ssprk3_stage(du0, du, dfl, dw, nv, extents, a, b, dt, du0)      # out is u0
    torch.cuda.synchronize()
    assert_bits_equal(to_host(du0), want, what="in place into u0")
    rhs = inputs.normal_f64(11, 0, u.size)
    du = to_dev(u)
    api.ssprk3_axpby(du, du, to_dev(rhs), nv, extents, a, b, dt, du)    # u0 = u = out
    torch.cuda.synchronize()
    assert_bits_equal(to_host(du), oracle.rk_axpby(u, u, rhs, a, b, dt), what="axpby in place")
    n = u.size
    big = torch.zeros(3 * n, dtype=torch.float64, device="cuda")
    before = api.launch_count()
    cases = [
        lambda: api.ssprk3_stage(big[:n], to_dev(u), dfl, dw, nv, extents, a, b, dt,
                                 big[8: 8 + n]),
        lambda: api.ssprk3_stage(to_dev(u0), big[:n], dfl, dw, nv, extents, a, b, dt,
                                 big[n - 1: 2 * n - 1]),
        lambda: api.ssprk3_stage(to_dev(u0), to_dev(u), dfl, dw, nv, extents, a, b, dt,
                                 dfl[1][:n]),
        lambda: api.ssprk3_axpby(to_dev(u0), to_dev(u), big[:n], nv, extents, a, b, dt,
                                 big[n // 2: n // 2 + n]),
    ]
    for case in cases:
        with pytest.raises(api.FvfError) as e:
            case()
        assert e.value.status == 6
    assert api.launch_count() == before
    with pytest.raises(api.FvfError) as e:
        api.ssprk3_stage(to_dev(u0), to_dev(u), dfl, dw, nv, extents, float("nan"), b, dt,
                         to_dev(u))
    assert e.value.status == 7
    torch.cuda.synchronize()


def test_full_ssprk3_step_201_cubed():
    """nv = 8 on 201^3 cells, x/y/z face fluxes N(0,1), inv_d = 1/d with
    d ~ U[0.5, 1.5]/201: the three stages of one step in place (stage s reads
    u^n and the previous stage, writes the stage over it), every element of
    every stage compared with the oracle."""
    torch = torch_cuda()
    extents, nv = (201, 201, 201), 8
    fl, w, u0, _ = _case(inputs.config_seed(11), extents, nv)
    dfl = [to_dev(f) for f in fl]
    dw = [to_dev(x) for x in w]
    du0 = to_dev(u0)
    du = to_dev(u0)
    want = u0
    dt = 1e-4
    for a, b in COEFS[:3]:
        api.ssprk3_stage(du0, du, dfl, dw, nv, extents, a, b, dt, du)
        torch.cuda.synchronize()
        want = oracle.ssprk3_stage(u0, want, fl, w, nv, extents, a, b, dt)
        assert_bits_equal(to_host(du), want, what=f"201^3 stage a={a}")


def test_stage_2d_4800x1200():
    """The 2D multi-variable case (nv = 7, 4800 x 1200, x and y fluxes): one
    fused stage, every element compared."""
    torch = torch_cuda()
    extents, nv = (4800, 1200, 1), 7
    fl, w, u0, u = _case(inputs.config_seed(12), extents, nv)
    fl[2] = None
    got = _gpu_stage(torch, u0, u, fl, w, nv, extents, 0.75, 0.25, 2e-5)
    assert_bits_equal(got, oracle.ssprk3_stage(u0, u, fl, w, nv, extents, 0.75, 0.25, 2e-5))


def test_wide_plane_64bit_indexing():
    """A plane of 2^31 cells (65536 x 32768 x 1, nv = 1) takes the 64-bit
    index path: the stage alone and fused with an x flux, on values given by
    a formula of the element index (built in place on the device, 52 GB at
    most), checked at sampled elements against the oracle on the same
    values."""
    torch = torch_cuda()
    n1, n2 = 65536, 32768
    extents, n = (n1, n2, 1), n1 * n2

    def ramp(count, mod, off, scale):
        t = torch.arange(count, dtype=torch.float64, device="cuda")
        return t.remainder_(mod).sub_(off).mul_(scale)

    u = ramp(n, 1000003.0, 500000.0, 1e-3)
    rhs = ramp(n, 999983.0, 499991.0, 2e-3)
    out = torch.empty_like(u)
    api.ssprk3_axpby(u, u, rhs, 1, extents, 0.75, 0.25, 0.3, out)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    s = np.concatenate([np.arange(4096), np.arange(n - 4096, n),
                        rng.integers(0, n, 1 << 15)]).astype(np.int64)
    sample = torch.from_numpy(s).cuda()
    us, rs = to_host(u[sample]), to_host(rhs[sample])
    assert_bits_equal(to_host(out[sample]), oracle.rk_axpby(us, us, rs, 0.75, 0.25, 0.3),
                      what="axpby 2^31")
    del rhs
    fx = ramp((n1 + 1) * n2, 999979.0, 499989.0, 1e-3)
    wx = torch.arange(n1, dtype=torch.float64, device="cuda").remainder_(7.0).mul_(0.125).add_(1.0)
    api.ssprk3_stage(u, u, [fx, None, None], [wx, None, None], 1, extents, 0.75, 0.25, 0.3, out)
    torch.cuda.synchronize()
    j, k = s % n1, s // n1
    lo = torch.from_numpy(j + (n1 + 1) * k).cuda()
    flo, fhi = to_host(fx[lo]), to_host(fx[lo + 1])
    wj = to_host(wx)[j]
    got = to_host(out[sample])
    # the oracle's x flux difference on one-cell rows, grouped by inverse width
    for wv in np.unique(wj):
        m = wj == wv
        faces = np.stack([flo[m], fhi[m]], axis=1).reshape(-1)
        term = oracle.advect_rhs(faces, np.array([wv]), 1, (1, int(m.sum()), 1), 0)
        assert_bits_equal(got[m], oracle.rk_axpby(us[m], us[m], term, 0.75, 0.25, 0.3),
                          what=f"stage 2^31 w={wv}")
