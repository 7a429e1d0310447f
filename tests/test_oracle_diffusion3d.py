"""Pins of the oracle's 3D 7-point diffusion against facts that do not come
from the oracle: exact one-step values of an impulse, the discrete eigenmode
decay factor, exact rational arithmetic on dyadic inputs, a worked FP32 value
that fixes the summation order, and the x-mirror symmetry.  CPU only."""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import inputs


def test_one_step_impulse_exact():
    """alpha = 1/8: the centre keeps 1 - 6/8, each of the six neighbours gets
    1/8, everything else stays 0 (all exact)."""
    u = np.zeros((7, 6, 5))
    u[3, 2, 2] = 1.0
    got = oracle.diffuse3d(u, 1, 0.125)
    want = np.zeros_like(u)
    want[3, 2, 2] = 0.25
    for dk, dj, di in ((1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1)):
        want[3 + dk, 2 + dj, 2 + di] = 0.125
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("shape,modes,steps", [((9, 11, 13), (1, 1, 1), 5),
                                               ((12, 10, 8), (2, 3, 1), 3)])
def test_eigenmode_decay(dtype, shape, modes, steps):
    """A product of sines vanishing on the boundary faces is an eigenvector of
    the update: each step multiplies it by 1 - 4 alpha (sx + sy + sz) with
    s = sin^2(p pi / (2 (n - 1))) per axis."""
    nz, ny, nx = shape
    pz, py, px = modes
    alpha = 0.1
    k, j, i = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
    phi = (np.sin(px * np.pi * i / (nx - 1)) * np.sin(py * np.pi * j / (ny - 1))
           * np.sin(pz * np.pi * k / (nz - 1)))
    phi[(i == 0) | (i == nx - 1) | (j == 0) | (j == ny - 1) | (k == 0) | (k == nz - 1)] = 0.0
    lam = 1.0 - 4.0 * alpha * sum(math.sin(p * math.pi / (2 * (n - 1))) ** 2
                                  for p, n in ((px, nx), (py, ny), (pz, nz)))
    got = oracle.diffuse3d(phi.astype(dtype), steps, alpha).astype(np.float64)
    want = lam ** steps * phi
    tol = (1e-13 if dtype == np.float64 else 3e-6) * steps
    assert np.max(np.abs(got - want)) < tol


def _exact_steps(u0, steps, alpha):
    """The update in exact rational arithmetic (edges written 0)."""
    nz, ny, nx = u0.shape
    a = Fraction(alpha)
    cur = [[[Fraction(float(u0[k, j, i])) for i in range(nx)] for j in range(ny)]
           for k in range(nz)]
    for _ in range(steps):
        nxt = [[[Fraction(0)] * nx for _ in range(ny)] for _ in range(nz)]
        for k in range(1, nz - 1):
            for j in range(1, ny - 1):
                for i in range(1, nx - 1):
                    c = cur[k][j][i]
                    s = (cur[k][j][i - 1] + cur[k][j][i + 1] + cur[k][j - 1][i]
                         + cur[k][j + 1][i] + cur[k - 1][j][i] + cur[k + 1][j][i])
                    nxt[k][j][i] = c + a * (s - 6 * c)
        cur = nxt
    return np.array([[[float(x) for x in row] for row in plane] for plane in cur])


def test_exact_on_dyadic_inputs_with_nonzero_edges():
    """Inputs k/16 with |k| < 64 (edges included, which the first step must
    zero) and alpha = 1/8 keep every intermediate exact in binary64 for two
    steps, so the oracle must equal exact rational arithmetic bit for bit;
    a wrong neighbour, weight or edge write breaks it."""
    shape = (5, 6, 7)
    bits = inputs.random_bits(21, 0, int(np.prod(shape)))
    u0 = ((bits % np.uint64(127)).astype(np.int64) - 63).astype(np.float64).reshape(shape) / 16.0
    for steps in (1, 2):
        got = oracle.diffuse3d(u0, steps, 0.125)
        assert np.array_equal(got, _exact_steps(u0, steps, 0.125)), steps


def test_summation_order_fp32_worked_value():
    """FP32, centre 0, W = 1 and the other five neighbours 2^-24: left to
    right every partial sum 1 + 2^-24 rounds back to 1 (ties to even), so the
    bracket is exactly 1 and the cell becomes fl32(alpha).  Any other order
    adds two of the small neighbours first and gives a larger bracket."""
    u = np.zeros((3, 3, 3), dtype=np.float32)
    tiny = np.float32(2.0 ** -24)
    u[1, 1, 0] = 1.0                      # W
    u[1, 1, 2] = tiny                     # E
    u[1, 0, 1] = u[1, 2, 1] = tiny        # S, N
    u[0, 1, 1] = u[2, 1, 1] = tiny        # B, T
    got = oracle.diffuse3d(u, 1, 0.1)
    assert got[1, 1, 1] == np.float32(0.1)


def test_x_mirror_symmetry_is_bitwise():
    """Mirroring i swaps W and E, whose sum is formed first and commutes
    exactly, so the result mirrors bit for bit."""
    shape = (6, 7, 9)
    u0 = inputs.uniform_f64(22, 0, int(np.prod(shape))).reshape(shape)
    a = oracle.diffuse3d(u0, 4, 0.1)
    b = oracle.diffuse3d(u0[:, :, ::-1].copy(), 4, 0.1)[:, :, ::-1]
    assert np.array_equal(a, b)


def test_stability_bound_and_mass_loss():
    """alpha <= 1/6 keeps a nonnegative field nonnegative and bounded by its
    maximum; with zero boundary faces the total never grows."""
    shape = (8, 9, 10)
    u0 = np.zeros(shape)
    u0[1:-1, 1:-1, 1:-1] = inputs.uniform_f64(23, 0, 6 * 7 * 8).reshape(6, 7, 8)
    masses = [u0.sum()]
    u = u0
    for _ in range(6):
        u = oracle.diffuse3d(u, 1, 1.0 / 6.0)
        assert u.min() >= 0.0 and u.max() <= u0.max()
        masses.append(u.sum())
    assert all(m1 <= m0 + 1e-12 for m0, m1 in zip(masses, masses[1:]))
