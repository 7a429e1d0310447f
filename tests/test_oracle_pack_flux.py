"""Pins of the CPU oracle's WENO pack and flux-difference source (MFC pull
request #2087, "Collapse only spatial loops in per-variable GPU kernels",
"Changes").

The expected values come from independent formulations (numpy slicing and
transposition of the Fortran-ordered boxes, coordinate-tagged fields), exact
special cases (constant and linear fluxes) and invariants (telescoping sums,
bit-for-bit copies of NaN payloads and signed zeros).
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import inputs

SHAPES = [((3, 4, 5), 1), ((3, 4, 5), 2), ((5, 4, 1), 2), ((6, 3, 2), 3), ((2, 7, 3), 1)]


def _box(flat, stored):
    """View a Fortran-ordered stored box as a numpy array indexed [l, k, j]."""
    N1, N2, N3 = stored
    return np.asarray(flat).reshape(N3, N2, N1)


def _numpy_pack(fields, extents, g, direction):
    """The pack written with numpy slices and transposes of [l, k, j] arrays."""
    n1, n2, n3 = extents
    st = inputs.stored_extents(extents, g)
    g1, g2, g3 = (g if n > 1 else 0 for n in extents)
    parts = []
    for f in fields:
        A = _box(f, st)
        if direction == 0:      # out[c, b, a] = A[c+g3, b+g2, a]
            S = A[g3:g3 + n3, g2:g2 + n2, :]
        elif direction == 1:    # out[c, b, a] = A[c+g3, a, b+g1]
            S = A[g3:g3 + n3, :, g1:g1 + n1].transpose(0, 2, 1)
        else:                   # out[c, b, a] = A[a, b+g2, c+g1]
            S = A[:, g2:g2 + n2, g1:g1 + n1].transpose(2, 1, 0)
        parts.append(np.ascontiguousarray(S).reshape(-1))
    return np.concatenate(parts)


@pytest.mark.parametrize("extents,g", SHAPES)
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3])
def test_pack_matches_numpy_formulation(extents, g, direction, nv):
    if extents[direction] == 1:
        pytest.skip("no sweep along an axis of extent 1")
    st = inputs.stored_extents(extents, g)
    fields = inputs.normal_fields(inputs.config_seed(0), nv, extents, g)
    got = oracle.weno_pack(fields, extents, g, direction)
    want = _numpy_pack(fields, extents, g, direction)
    assert got.shape == want.shape
    assert np.array_equal(got.view(np.uint64), want.view(np.uint64))
    M = oracle.pack_extents(extents, g, direction)
    assert got.size == M[0] * M[1] * M[2] * nv
    assert st[direction] == M[0]


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_pack_coordinate_tags(direction):
    """Each source element carries its own (i, j, k, l) as an exact number;
    decoding the output must give the swept axis (with its ghosts) first, the
    other axes' interior cells next, and the variable slowest."""
    extents, g = (4, 5, 6), 2
    n1, n2, n3 = extents
    N1, N2, N3 = inputs.stored_extents(extents, g)
    nv = 3
    fields = []
    for i in range(nv):
        l, k, j = np.meshgrid(np.arange(N3), np.arange(N2), np.arange(N1), indexing="ij")
        fields.append((i * 1e9 + j * 1e6 + k * 1e3 + l).astype(np.float64).reshape(-1))
    out = oracle.weno_pack(fields, extents, g, direction)
    M1, M2, M3 = oracle.pack_extents(extents, g, direction)
    for i, c, b, a in itertools.product(range(nv), range(M3), range(M2), range(M1)):
        val = int(out[a + M1 * (b + M2 * (c + M3 * i))])
        ti, r = divmod(val, 10**9)
        tj, r = divmod(r, 10**6)
        tk, tl = divmod(r, 10**3)
        if direction == 0:
            want = (a, b + g, c + g)
        elif direction == 1:
            want = (b + g, a, c + g)
        else:
            want = (c + g, b + g, a)
        assert (ti, tj, tk, tl) == (i, *want)


def test_pack_copies_bits_exactly():
    """NaN payloads, signed zeros, infinities and subnormals survive the pack
    bit for bit (it is a copy, not arithmetic)."""
    extents, g = (3, 4, 5), 1
    n = int(np.prod(inputs.stored_extents(extents, g)))
    bits = inputs.random_bits(7, 0, n)
    special = np.array([0x7FF8000000000001, 0xFFF0000000000000, 0x8000000000000000,
                        0x0000000000000001, 0x7FF4DEADBEEF0000, 0x7FF0000000000000],
                       dtype=np.uint64)
    bits[: special.size] = special
    bits[-special.size:] = special
    for direction in range(3):
        f = bits.view(np.float64)
        got = oracle.weno_pack([f], extents, g, direction)
        want = _numpy_pack([f], extents, g, direction)
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64))


def test_pack_round_trip_recovers_sub_box():
    """Scattering the pack back through the inverse permutation restores the
    swept-axis-with-ghosts by interior-transverse sub-box exactly."""
    extents, g = (5, 6, 7), 2
    st = inputs.stored_extents(extents, g)
    f = inputs.normal_fields(3, 1, extents, g)[0]
    A = _box(f, st)
    for direction in range(3):
        out = oracle.weno_pack([f], extents, g, direction)
        M1, M2, M3 = oracle.pack_extents(extents, g, direction)
        O = out.reshape(M3, M2, M1)
        if direction == 0:
            back = O
            ref = A[g:-g, g:-g, :]
        elif direction == 1:
            back = O.transpose(0, 2, 1)
            ref = A[g:-g, :, g:-g]
        else:
            back = O.transpose(2, 1, 0)
            ref = A[:, g:-g, g:-g]
        assert np.array_equal(back, ref)


# ---------------------------------------------------------------------------
# Flux difference
# ---------------------------------------------------------------------------

def _numpy_rhs(flux, inv_d, nv, extents, direction):
    """The flux difference with numpy differences along the swept axis of a
    [i, l, k, j] array: rhs = inv_d * (F[low face] - F[high face])."""
    n1, n2, n3 = extents
    F1, F2, F3 = oracle.flux_extents(extents, direction)
    F = np.asarray(flux).reshape(nv, F3, F2, F1)
    if direction == 0:
        return (inv_d[None, None, None, :] * (F[..., :-1] - F[..., 1:])).reshape(-1)
    if direction == 1:
        return (inv_d[None, None, :, None] * (F[:, :, :-1, :] - F[:, :, 1:, :])).reshape(-1)
    return (inv_d[None, :, None, None] * (F[:, :-1] - F[:, 1:])).reshape(-1)


@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (1, 6, 2), (7, 1, 3)])
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3])
def test_rhs_matches_numpy_formulation(extents, direction, nv):
    seed = inputs.config_seed(0)
    flux = inputs.face_fluxes(seed, nv, extents, direction)
    inv_d = inputs.inverse_spacing(seed, extents[direction], stream=200 + direction)
    got = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
    want = _numpy_rhs(flux, inv_d, nv, extents, direction)
    assert np.array_equal(got.view(np.uint64), want.view(np.uint64))


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_rhs_constant_flux_is_positive_zero(direction):
    """A constant flux has no difference: rhs is +0.0 exactly (inv_d > 0)."""
    extents, nv = (4, 5, 6), 2
    F = np.full(int(np.prod(oracle.flux_extents(extents, direction))) * nv, 3.25)
    inv_d = inputs.inverse_spacing(1, extents[direction])
    rhs = oracle.advect_rhs(F, inv_d, nv, extents, direction)
    assert np.all(rhs.view(np.uint64) == 0)


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_rhs_linear_flux_gives_minus_inv_d(direction):
    """F(f) = f along the swept axis (face f stored at position f + 1):
    F(c-1) - F(c) = -1 exactly, so rhs = -inv_d(c) exactly; the sign fixes
    which face is subtracted from which."""
    extents, nv = (4, 5, 6), 2
    F1, F2, F3 = oracle.flux_extents(extents, direction)
    l, k, j = np.meshgrid(np.arange(F3), np.arange(F2), np.arange(F1), indexing="ij")
    pos = (j, k, l)[direction] - 1.0
    F = np.tile(pos.reshape(-1), nv)
    inv_d = inputs.inverse_spacing(5, extents[direction])
    rhs = oracle.advect_rhs(F, inv_d, nv, extents, direction)
    n1, n2, n3 = extents
    R = rhs.reshape(nv, n3, n2, n1)
    shape = [1, 1, 1, 1]
    shape[3 - direction] = -1
    assert np.array_equal(R, np.broadcast_to(-inv_d.reshape(shape), R.shape))


def test_rhs_telescopes():
    """Summing rhs/inv_d along the swept axis gives F(-1) - F(n-1) up to
    rounding (the interior faces cancel)."""
    extents, nv = (9, 4, 3), 2
    flux = inputs.face_fluxes(11, nv, extents, 0)
    inv_d = inputs.inverse_spacing(11, 9)
    rhs = oracle.advect_rhs(flux, inv_d, nv, extents, 0).reshape(nv, 3, 4, 9)
    F = flux.reshape(nv, 3, 4, 10)
    s = np.array([[[math.fsum((rhs[i, l, k, :] / inv_d).tolist()) for k in range(4)]
                   for l in range(3)] for i in range(nv)])
    assert np.allclose(s, F[..., 0] - F[..., -1], rtol=0, atol=1e-13)


def test_multivar_sequence_shapes():
    """The 2D multi-variable sequence (pack x, pack y, rhs x, rhs y) on a
    small box returns outputs of the sizes the layouts imply."""
    extents, g, nv = (12, 8, 1), 2, 7
    seed = inputs.config_seed(5)
    fields = inputs.multivar_fields_2d(seed, extents, g)
    fx = inputs.face_fluxes(seed, nv, extents, 0)
    fy = inputs.face_fluxes(seed, nv, extents, 1)
    wx = inputs.inverse_spacing(seed, 12, stream=200)
    wy = inputs.inverse_spacing(seed, 8, stream=201)
    px, py, rx, ry = oracle.multivar_sweep_2d(fields, fx, fy, wx, wy, nv, extents, g)
    assert px.size == 16 * 8 * 7 and py.size == 12 * 12 * 7
    assert rx.size == ry.size == 12 * 8 * 7
    assert np.all(fields[5] >= 0) and np.all(fields[5] < 1)
    assert np.all(fields[0] > 0)


# ---------------------------------------------------------------------------
# Accumulating flux difference and the directional flux copy (unpack)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (7, 1, 3)])
@pytest.mark.parametrize("direction", [0, 1, 2])
def test_rhs_add_matches_numpy_formulation(extents, direction):
    """rhs_new = rhs_old + inv_d*(F(c-1) - F(c)), each operation rounded once
    (numpy float64, no contraction)."""
    nv = 3
    seed = inputs.config_seed(0)
    flux = inputs.face_fluxes(seed, nv, extents, direction)
    inv_d = inputs.inverse_spacing(seed, extents[direction], stream=210 + direction)
    old = inputs.normal_f64(seed, 300 + direction, int(np.prod(extents)) * nv)
    got = oracle.advect_rhs_add(flux, inv_d, nv, extents, direction, old)
    want = old + _numpy_rhs(flux, inv_d, nv, extents, direction)
    assert np.array_equal(got.view(np.uint64), want.view(np.uint64))


def test_rhs_add_into_zero_is_assignment():
    """Accumulating into +0 gives the assigned term, except that a -0 term
    becomes +0 (+0 + -0 = +0 under round to nearest)."""
    extents, nv = (6, 5, 4), 2
    for direction in range(3):
        flux = inputs.face_fluxes(3, nv, extents, direction)
        flux[::9] = 1.5                     # some equal faces: zero differences
        inv_d = inputs.inverse_spacing(3, extents[direction])
        zero = np.zeros(int(np.prod(extents)) * nv)
        acc = oracle.advect_rhs_add(flux, inv_d, nv, extents, direction, zero)
        asg = oracle.advect_rhs(flux, inv_d, nv, extents, direction)
        assert np.array_equal(acc, asg)
        assert np.array_equal(acc.view(np.uint64), np.where(asg == 0, 0.0, asg).view(np.uint64))


def test_rhs_add_builds_two_direction_sum():
    """Linear fluxes along x and along y, accumulated into zero: each cell
    holds (-inv_dx) + (-inv_dy), rounded once."""
    extents, nv = (4, 5, 1), 2
    wx = inputs.inverse_spacing(8, 4)
    wy = inputs.inverse_spacing(9, 5, stream=201)
    rhs = np.zeros(4 * 5 * nv)
    for direction, w in ((0, wx), (1, wy)):
        F1, F2, F3 = oracle.flux_extents(extents, direction)
        l, k, j = np.meshgrid(np.arange(F3), np.arange(F2), np.arange(F1), indexing="ij")
        F = np.tile(((j, k, l)[direction] - 1.0).reshape(-1), nv)
        rhs = oracle.advect_rhs_add(F, w, nv, extents, direction, rhs)
    R = rhs.reshape(nv, 1, 5, 4)
    want = (-wx)[None, None, None, :] + (-wy)[None, None, :, None]
    assert np.array_equal(R, np.broadcast_to(want, R.shape))


def _numpy_unpack(src, nv, extents, direction):
    """Sweep frame -> physical frame with numpy transposes of [i, c, b, a]
    arrays (a = swept axis)."""
    S = oracle.sweep_flux_extents(extents, direction)
    A = np.asarray(src).reshape(nv, S[2], S[1], S[0])      # [i, c, b, a]
    if direction == 0:
        P = A                                               # out[i, l, k, f] = in[i, l, k, f]
    elif direction == 1:
        P = A.transpose(0, 1, 3, 2)                         # out[i, l, f, j] = in[i, l, j, f]
    else:
        P = A.transpose(0, 3, 2, 1)                         # out[i, f, k, j] = in[i, j, k, f]
    return np.ascontiguousarray(P).reshape(-1)


@pytest.mark.parametrize("extents", [(3, 4, 5), (5, 4, 1), (1, 6, 2), (7, 1, 3)])
@pytest.mark.parametrize("direction", [0, 1, 2])
def test_flux_unpack_matches_numpy_formulation(extents, direction):
    nv = 3
    src = inputs.normal_f64(4, direction, int(np.prod(oracle.sweep_flux_extents(extents, direction))) * nv)
    got = oracle.flux_unpack(src, nv, extents, direction)
    assert np.array_equal(got.view(np.uint64), _numpy_unpack(src, nv, extents, direction).view(np.uint64))


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_flux_unpack_coordinate_tags(direction):
    """Each sweep-frame element carries (i, a, b, c); the physical element
    (j, k, l, i) must hold the tag of the face it is: a = the swept-axis face
    index, b and c the transverse cells in the sweep frame's order."""
    extents, nv = (4, 5, 6), 2
    S = oracle.sweep_flux_extents(extents, direction)
    c, b, a = np.meshgrid(np.arange(S[2]), np.arange(S[1]), np.arange(S[0]), indexing="ij")
    src = np.concatenate([(i * 1e9 + a * 1e6 + b * 1e3 + c).astype(np.float64).reshape(-1)
                          for i in range(nv)])
    out = oracle.flux_unpack(src, nv, extents, direction)
    F1, F2, F3 = oracle.flux_extents(extents, direction)
    for i, l, k, j in itertools.product(range(nv), range(F3), range(F2), range(F1)):
        val = int(out[j + F1 * (k + F2 * (l + F3 * i))])
        ti, r = divmod(val, 10**9)
        ta, r = divmod(r, 10**6)
        tb, tc = divmod(r, 10**3)
        want = [(j, k, l), (k, j, l), (l, k, j)][direction]
        assert (ti, ta, tb, tc) == (i, *want)


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_flux_unpack_inverts_the_pack_permutation(direction):
    """A physical face array packed along its direction (ghost width 0, the
    face-extended extents as the box) and unpacked again is unchanged."""
    extents, nv = (5, 6, 7), 3
    fe = oracle.flux_extents(extents, direction)
    phys = inputs.normal_f64(12, direction, int(np.prod(fe)) * nv)
    fields = [phys[i * int(np.prod(fe)):(i + 1) * int(np.prod(fe))] for i in range(nv)]
    sweep = oracle.weno_pack(fields, fe, 0, direction)
    back = oracle.flux_unpack(sweep, nv, extents, direction)
    assert np.array_equal(back.view(np.uint64), phys.view(np.uint64))


# ---------------------------------------------------------------------------
# Conservative-variable copy (and the pack fused with it)
# ---------------------------------------------------------------------------

def test_fields_copy_is_bitwise_identity():
    """Every element of every stored box, ghosts included, is copied bit for
    bit (NaN payloads, signed zeros and subnormals too)."""
    extents, g, nv = (5, 4, 3), 2, 3
    n = int(np.prod(inputs.stored_extents(extents, g)))
    fields = [inputs.random_bits(31, i, n).view(np.float64) for i in range(nv)]
    fields[0][:4] = np.array([0x7FF4000000000001, 0x8000000000000000, 1, 0x7FF0000000000000],
                             dtype=np.uint64).view(np.float64)
    copies = oracle.fields_copy(fields, extents, g)
    for f, c in zip(fields, copies):
        assert c.size == n
        assert np.array_equal(f.view(np.uint64), c.view(np.uint64))


def test_pack_copy_is_pack_and_copy():
    extents, g, nv = (6, 5, 4), 2, 2
    fields = inputs.normal_fields(5, nv, extents, g)
    for direction in range(3):
        packed, copies = oracle.weno_pack_copy(fields, extents, g, direction)
        assert np.array_equal(packed, _numpy_pack(fields, extents, g, direction))
        assert all(np.array_equal(a, b) for a, b in zip(copies, fields))


# ---------------------------------------------------------------------------
# FP32 forms of the pack and of the flux difference
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("direction", [0, 1, 2])
def test_pack_f32_coordinate_tags(direction):
    """FP32 fields carrying their own (i, j, k, l) as exact binary32 integers
    (below 2^24): the FP32 pack must place them as the mapping states."""
    extents, g = (4, 5, 6), 2
    N1, N2, N3 = inputs.stored_extents(extents, g)
    nv = 3
    fields = []
    for i in range(nv):
        l, k, j = np.meshgrid(np.arange(N3), np.arange(N2), np.arange(N1), indexing="ij")
        fields.append((i * 100000 + j * 1000 + k * 32 + l).astype(np.float32).reshape(-1))
    out = oracle.weno_pack(fields, extents, g, direction)
    assert out.dtype == np.float32
    M1, M2, M3 = oracle.pack_extents(extents, g, direction)
    for i, c, b, a in itertools.product(range(nv), range(M3), range(M2), range(M1)):
        val = int(out[a + M1 * (b + M2 * (c + M3 * i))])
        ti, r = divmod(val, 100000)
        tj, r = divmod(r, 1000)
        tk, tl = divmod(r, 32)
        want = [(a, b + g, c + g), (b + g, a, c + g), (c + g, b + g, a)][direction]
        assert (ti, tj, tk, tl) == (i,) + want


def test_pack_f32_is_the_fp64_pack_of_the_same_values():
    """Widening binary32 to binary64 is exact, so packing in FP32 then
    widening equals widening then packing in FP64 (NaN payloads aside, the
    values are random normals here)."""
    extents, g = (7, 6, 5), 3
    fields = inputs.normal_fields(12, 4, extents, g)
    f32 = [f.astype(np.float32) for f in fields]
    for direction in range(3):
        a = oracle.weno_pack(f32, extents, g, direction).astype(np.float64)
        b = oracle.weno_pack([f.astype(np.float64) for f in f32], extents, g, direction)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_rhs_f32_linear_and_constant_flux(direction):
    """FP32: F(f) = f gives exactly -inv_d; a constant flux gives +0."""
    extents, nv = (4, 5, 6), 2
    F1, F2, F3 = oracle.flux_extents(extents, direction)
    l, k, j = np.meshgrid(np.arange(F3), np.arange(F2), np.arange(F1), indexing="ij")
    pos = ((j, k, l)[direction] - 1.0).astype(np.float32)
    F = np.tile(pos.reshape(-1), nv)
    inv_d = inputs.inverse_spacing(5, extents[direction]).astype(np.float32)
    rhs = oracle.advect_rhs(F, inv_d, nv, extents, direction)
    assert rhs.dtype == np.float32
    n1, n2, n3 = extents
    R = rhs.reshape(nv, n3, n2, n1)
    shape = [1, 1, 1, 1]
    shape[3 - direction] = -1
    assert np.array_equal(R, np.broadcast_to(-inv_d.reshape(shape), R.shape))
    const = oracle.advect_rhs(np.full_like(F, np.float32(2.5)), inv_d, nv, extents, direction)
    assert np.all(const == 0) and not np.signbit(const).any()


def test_rhs_f32_is_the_rounded_exact_value():
    """For binary32 inputs of moderate range the difference and the product
    are exact in binary64, so each FP32 operation equals the binary64 result
    rounded once to binary32: the FP32 term must be
    f32(f64(w) * f64(f32(f64(lo) - f64(hi)))), assigned or added."""
    extents, nv = (9, 8, 7), 3
    for direction in range(3):
        flux = inputs.face_fluxes(13, nv, extents, direction).astype(np.float32)
        w = inputs.inverse_spacing(13, extents[direction], stream=200 + direction).astype(np.float32)
        F = flux.reshape((nv,) + tuple(oracle.flux_extents(extents, direction))[::-1])
        lo = np.take(F, np.arange(extents[direction]), axis=3 - direction).astype(np.float64)
        hi = np.take(F, np.arange(1, extents[direction] + 1), axis=3 - direction).astype(np.float64)
        shape = [1, 1, 1, 1]
        shape[3 - direction] = -1
        diff = (lo - hi).astype(np.float32).astype(np.float64)
        term = (w.astype(np.float64).reshape(shape) * diff).astype(np.float32)
        got = oracle.advect_rhs(flux, w, nv, extents, direction)
        assert np.array_equal(got, term.reshape(-1))
        base = inputs.normal_f64(14, direction, got.size).astype(np.float32)
        acc = oracle.advect_rhs_add(flux, w, nv, extents, direction, base)
        want = (base.astype(np.float64) + term.reshape(-1).astype(np.float64)).astype(np.float32)
        assert np.array_equal(acc, want)
