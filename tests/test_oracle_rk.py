"""Pins of the oracle's SSPRK3 stage update (axpby) and of the stage fused
with the flux difference, against facts that do not come from the oracle:
values worked by hand in exact binary arithmetic, the closed form of SSPRK3
on a linear equation, identities of the coefficients and the telescoping of
the flux differences.  CPU only."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import inputs

# Shu-Osher SSPRK3 coefficients, written out here independently of the
# oracle's own table: stage s computes a*u^n + b*(u + dt*L(u)).
STAGES = [(0.0, 1.0), (0.75, 0.25), (1.0 / 3.0, 2.0 / 3.0)]


def test_stage_table_is_shu_osher():
    assert oracle.SSPRK3_STAGES == tuple(STAGES)
    for a, b in STAGES:  # consistency: a constant state stays constant
        assert a + b == pytest.approx(1.0, abs=1e-16)


@pytest.mark.parametrize("u0,u,rhs,dt,a,b,want", [
    # t = u + dt*rhs, then a*u0 + b*t; every value below is exact in binary64
    (1.0, 2.0, 4.0, 0.5, 0.75, 0.25, 1.75),       # t = 4, 0.75 + 1
    (5.0, 3.0, -8.0, 0.25, 0.0, 1.0, 1.0),        # t = 1, 0*5 + 1
    (3.0, 1.5, 1.0, 1.5, 1.0 / 3.0, 2.0 / 3.0, 3.0),  # t = 3; fl(1/3)*3 = 1, fl(2/3)*3 = 2 (ties to even)
    (-2.0, 0.5, 6.0, -0.125, 0.75, 0.25, -1.5625),    # t = -0.25, -1.5 - 0.0625
    (8.0, 8.0, 0.0, 1.0, 0.0, 1.0, 8.0),
])
def test_axpby_worked_values(u0, u, rhs, dt, a, b, want):
    got = oracle.rk_axpby(np.array([u0]), np.array([u]), np.array([rhs]), a, b, dt)
    assert got[0] == want


def test_axpby_coefficient_identities():
    """a = 1, b = 0 returns u0; a = 0, b = 1 with dt = 0 returns u (nonzero
    finite entries, so no signed-zero corner)."""
    n = 4096
    u0 = inputs.normal_f64(11, 0, n) + 3.0
    u = inputs.normal_f64(11, 1, n) - 3.0
    rhs = inputs.normal_f64(11, 2, n)
    assert np.array_equal(oracle.rk_axpby(u0, u, rhs, 1.0, 0.0, 0.7), u0)
    assert np.array_equal(oracle.rk_axpby(u0, u, rhs, 0.0, 1.0, 0.0), u)


def _ssprk3_linear(u_n, lam, dt):
    """Three stages on u' = lam*u, the rhs formed from each stage's state."""
    u = u_n
    for a, b in STAGES:
        u = oracle.rk_axpby(u_n, u, lam * u, a, b, dt)
    return u


@pytest.mark.parametrize("z", [-0.1, -0.5, -1.0, -2.0, -2.5, 0.3])
def test_ssprk3_closed_form_on_linear_equation(z):
    """On u' = lam*u SSPRK3 multiplies u^n by 1 + z + z^2/2 + z^3/6 with
    z = lam*dt (it is third order and, for a linear equation, equals the
    Taylor polynomial); a wrong coefficient, a swapped u^n/u or a dropped dt
    changes the polynomial."""
    n = 2048
    u_n = inputs.normal_f64(12, 0, n)
    dt = 0.375
    lam = z / dt
    got = _ssprk3_linear(u_n, lam, dt)
    p = 1.0 + z + z * z / 2.0 + z ** 3 / 6.0
    want = p * u_n
    scale = np.abs(u_n) * (1.0 + abs(z) + z * z / 2 + abs(z) ** 3 / 6)
    assert np.all(np.abs(got - want) <= 16 * np.finfo(float).eps * scale + 1e-300)


def test_ssprk3_is_third_order():
    """Halving dt divides the one-step error against exp(z) by about 16
    (local error O(dt^4))."""
    u_n = np.array([1.0])
    lam = -1.3
    errs = []
    for dt in (0.2, 0.1, 0.05):
        errs.append(abs(_ssprk3_linear(u_n, lam, dt)[0] - math.exp(lam * dt)))
    assert 12 < errs[0] / errs[1] < 20 and 12 < errs[1] / errs[2] < 20


# ---------------------------------------------------------------------------
# Stage fused with the flux difference
# ---------------------------------------------------------------------------

def _linear_faces(extents, direction, slope, nv):
    """Face array of one direction whose value at face f (-1 <= f <= n-1)
    along the swept axis is slope*f, for every variable."""
    fe = oracle.flux_extents(extents, direction)
    f = np.arange(fe[direction], dtype=np.float64) - 1.0
    shape = [1, 1, 1]
    shape[direction] = fe[direction]
    face = np.broadcast_to((slope * f).reshape(shape[::-1]), fe[::-1])
    return np.ascontiguousarray(np.broadcast_to(face, (nv,) + tuple(fe[::-1]))).reshape(-1)


def test_stage_linear_fluxes_worked_value():
    """Fluxes slope_d * f along each axis give rhs = -(1*2 + 2*4 + 3*0.5) =
    -11.5 with inverse spacings 2, 4, 0.5; with u = 1, u0 = 2, dt = 0.25,
    a = 0.75, b = 0.25: t = 1 - 2.875 = -1.875, out = 1.5 - 0.46875 =
    1.03125, all exact."""
    extents, nv = (5, 4, 3), 2
    fl = [_linear_faces(extents, d, s, nv) for d, s in ((0, 1.0), (1, 2.0), (2, 3.0))]
    w = [np.full(extents[d], v) for d, v in ((0, 2.0), (1, 4.0), (2, 0.5))]
    n = int(np.prod(extents)) * nv
    got = oracle.ssprk3_stage(np.full(n, 2.0), np.ones(n), fl, w, nv, extents, 0.75, 0.25, 0.25)
    assert np.all(got == 1.03125)
    # x only: rhs = -2, t = 0.5, out = 1.5 + 0.125
    got = oracle.ssprk3_stage(np.full(n, 2.0), np.ones(n), [fl[0], None, None], w, nv, extents,
                              0.75, 0.25, 0.25)
    assert np.all(got == 1.625)


def test_stage_conserves_with_telescoping_fluxes():
    """Summed over a row with cell widths d = 1/inv_d, d*rhs telescopes to
    F(-1) - F(n-1): so sum d*(out - a*u0 - b*u) = b*dt*(F(-1) - F(n-1)) up
    to rounding."""
    extents, nv = (40, 3, 2), 1
    seed = 77
    fl = [inputs.face_fluxes(seed, nv, extents, 0), None, None]
    w = [1.0 / (0.5 + inputs.uniform_f64(seed, 3, extents[0]))]
    n = int(np.prod(extents))
    u0 = inputs.normal_f64(seed, 4, n)
    u = inputs.normal_f64(seed, 5, n)
    a, b, dt = 0.75, 0.25, 0.01
    out = oracle.ssprk3_stage(u0, u, fl, w, nv, extents, a, b, dt)
    F = fl[0].reshape(extents[2], extents[1], extents[0] + 1)
    d = 1.0 / w[0]
    lhs = ((out - a * u0 - b * u).reshape(extents[2], extents[1], extents[0]) * d).sum(axis=2)
    rhs = b * dt * (F[:, :, 0] - F[:, :, -1])
    assert np.allclose(lhs, rhs, rtol=1e-9, atol=1e-12)


def test_stage_is_rhs_then_axpby():
    """The fused stage equals the flux-difference rhs followed by the stage
    update, for every choice of present directions."""
    extents, nv = (6, 5, 4), 3
    seed = 78
    fl = [inputs.face_fluxes(seed, nv, extents, d) for d in range(3)]
    w = [inputs.inverse_spacing(seed, extents[d], stream=200 + d) for d in range(3)]
    n = int(np.prod(extents)) * nv
    u0, u = inputs.normal_f64(seed, 6, n), inputs.normal_f64(seed, 7, n)
    for present in ((0,), (0, 1), (0, 2), (0, 1, 2)):
        f = [fl[d] if d in present else None for d in range(3)]
        rhs = oracle.advect_rhs(fl[0], w[0], nv, extents, 0)
        for d in present[1:]:
            rhs = oracle.advect_rhs_add(fl[d], w[d], nv, extents, d, rhs)
        for a, b in STAGES:
            got = oracle.ssprk3_stage(u0, u, f, w, nv, extents, a, b, 0.3)
            assert np.array_equal(got, oracle.rk_axpby(u0, u, rhs, a, b, 0.3))
