"""Property tests of the oracle over random shapes (hypothesis; skipped where
it is not installed): the C oracle's pack, flux difference and unpack agree
with their numpy slice-and-transpose formulations, and the 2D/3D diffusion
keep the properties the pages fix (zero edges, the x-mirror symmetry, the
maximum principle for alpha within the stability bound).  CPU only."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import tests.test_oracle_pack_flux as P
from finite_volume_field_gb300 import inputs

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

extent = st.integers(min_value=1, max_value=9)
ghost = st.integers(min_value=0, max_value=3)
direction = st.integers(min_value=0, max_value=2)
nvars = st.integers(min_value=1, max_value=4)
seed = st.integers(min_value=0, max_value=2 ** 31 - 1)


@settings(max_examples=60, deadline=None)
@given(n1=extent, n2=extent, n3=extent, g=ghost, d=direction, nv=nvars, s=seed)
def test_pack_matches_numpy(n1, n2, n3, g, d, nv, s):
    extents = (n1, n2, n3)
    fields = inputs.normal_fields(s, nv, extents, g)
    assert np.array_equal(oracle.weno_pack(fields, extents, g, d),
                          P._numpy_pack(fields, extents, g, d))
    f32 = [f.astype(np.float32) for f in fields]
    assert np.array_equal(oracle.weno_pack(f32, extents, g, d).astype(np.float64),
                          P._numpy_pack([f.astype(np.float64) for f in f32], extents, g, d))


@settings(max_examples=60, deadline=None)
@given(n1=extent, n2=extent, n3=extent, d=direction, nv=nvars, s=seed)
def test_flux_difference_and_unpack_match_numpy(n1, n2, n3, d, nv, s):
    extents = (n1, n2, n3)
    flux = inputs.face_fluxes(s, nv, extents, d)
    w = inputs.inverse_spacing(s, extents[d], stream=200 + d)
    assert np.array_equal(oracle.advect_rhs(flux, w, nv, extents, d),
                          P._numpy_rhs(flux, w, nv, extents, d))
    sweep = inputs.normal_f64(s + 1, 0, int(np.prod(oracle.sweep_flux_extents(extents, d))) * nv)
    assert np.array_equal(oracle.flux_unpack(sweep, nv, extents, d),
                          P._numpy_unpack(sweep, nv, extents, d))


@settings(max_examples=40, deadline=None)
@given(nx=st.integers(3, 24), ny=st.integers(3, 24), steps=st.integers(1, 6), s=seed,
       f32=st.booleans())
def test_diffusion_2d_properties(nx, ny, steps, s, f32):
    dt = np.float32 if f32 else np.float64
    u0 = inputs.uniform_f64(s, 0, nx * ny).reshape(ny, nx).astype(dt)
    u = oracle.diffuse2d(u0, steps, 0.25)
    assert not u[0].any() and not u[-1].any() and not u[:, 0].any() and not u[:, -1].any()
    assert u.min() >= 0 and u.max() <= u0.max()          # maximum principle, alpha = 1/4
    m = oracle.diffuse2d(u0[:, ::-1].copy(), steps, 0.25)[:, ::-1]
    assert np.array_equal(u, m)                          # W + E commutes exactly


@settings(max_examples=30, deadline=None)
@given(nx=st.integers(3, 12), ny=st.integers(3, 12), nz=st.integers(3, 12),
       steps=st.integers(1, 4), s=seed)
def test_diffusion_3d_properties(nx, ny, nz, steps, s):
    u0 = inputs.uniform_f64(s, 0, nx * ny * nz).reshape(nz, ny, nx)
    u = oracle.diffuse3d(u0, steps, 1.0 / 6.0)
    for face in (u[0], u[-1], u[:, 0], u[:, -1], u[:, :, 0], u[:, :, -1]):
        assert not face.any()
    assert u.min() >= 0 and u.max() <= u0.max()
    m = oracle.diffuse3d(u0[:, :, ::-1].copy(), steps, 1.0 / 6.0)[:, :, ::-1]
    assert np.array_equal(u, m)
