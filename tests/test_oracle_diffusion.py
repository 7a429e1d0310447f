"""Pins of the CPU oracle's 2D diffusion against what the Qiita page
("Fortran 2018 GPU acceleration, part 3") and the mathematics fix.

None of these checks reuses the oracle's own code: the expected values come
from the page's printed worked example (tests/golden), exact rational
arithmetic (fractions.Fraction), closed forms of the centre-impulse solution,
or invariants of the update.
"""
from __future__ import annotations

import math
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import inputs

GOLDEN = Path(__file__).parent / "golden"
ALPHA64 = Fraction(0.1)                            # the binary value of the double 0.1
ALPHA32 = Fraction(float(np.float32(0.1)))         # the binary value of 0.1_real32


def _read_golden(name):
    vals = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        vals[k] = v
    return vals


# ---------------------------------------------------------------------------
# The page's printed worked example (section 8.2)
# ---------------------------------------------------------------------------

def test_printed_fp32_vs_fp64_table():
    """Qiita section 8.2: FP32 vs FP64 CPU runs, 31 x 27, 32 steps.  Pins the
    operation order ((((W+E)+S)+N) - 4c), the absence of FMA contraction and
    round-to-nearest: other orders or a fused c + alpha*t change the printed
    digits."""
    g = _read_golden("qiita_fp32_vs_fp64_31x27_32steps.txt")
    nx, ny, steps = int(g["nx"]), int(g["ny"]), int(g["steps"])
    u64 = oracle.diffuse2d(oracle.centre_impulse(nx, ny, np.float64), steps)
    u32 = oracle.diffuse2d(oracle.centre_impulse(nx, ny, np.float32), steps)
    m = oracle.compare_fields(u64, u32, atol=float(g["atol"]), rtol=float(g["rtol"]))
    for key in ("max_abs", "relative_l2", "mass_difference"):
        assert f"{m[key]:.6e}" == g[key], (key, m[key], g[key])
    assert m["cells"] == int(g["cells"])
    assert m["failures"] == int(g["failures"])


def test_physical_checks_pass_on_worked_example():
    """Appendix A's print_summary checks (finite, bounds, mass) hold for both
    precisions of the worked example."""
    for dt in (np.float32, np.float64):
        u = oracle.diffuse2d(oracle.centre_impulse(31, 27, dt), 32)
        assert oracle.physical_check(u)["ok"]


# ---------------------------------------------------------------------------
# One step from the centre impulse
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_one_step_impulse(dt):
    """After one step the centre holds 1 - 4*alpha = 0.6 and its four
    neighbours alpha = 0.1 (Qiita section 3), bitwise in each precision;
    every other cell is zero."""
    u = oracle.diffuse2d(oracle.centre_impulse(64, 64, dt), 1)
    ci, cj = 31, 31  # 0-based centre of 64x64, the 1-based (32, 32)
    assert u[cj, ci] == dt(0.6)
    for dj, di in ((0, 1), (0, -1), (1, 0), (-1, 0)):
        assert u[cj + dj, ci + di] == dt(0.1)
    mask = np.ones_like(u, dtype=bool)
    mask[cj, ci] = False
    for dj, di in ((0, 1), (0, -1), (1, 0), (-1, 0)):
        mask[cj + dj, ci + di] = False
    assert np.all(u[mask] == 0)


def test_centre_convention_64():
    """The 1-based centre ((nx+1)/2, (ny+1)/2) of a 64x64 grid is (32, 32),
    i.e. 0-based (31, 31)."""
    u = oracle.centre_impulse(64, 64)
    assert u[31, 31] == 1.0 and u.sum() == 1.0


# ---------------------------------------------------------------------------
# Closed form of the centre-impulse solution on an unbounded grid
# ---------------------------------------------------------------------------

def _closed_form(a: int, b: int, n: int, alpha: Fraction) -> Fraction:
    """Value at offset (a, b) from the impulse after n steps on an unbounded
    grid: the coefficient of x^a y^b in ((1-4alpha) + alpha(x + 1/x + y + 1/y))^n.
    With x = pq, y = p/q the bracket factors as (p + 1/p)(q + 1/q), so the
    coefficient of x^a y^b in (x + 1/x + y + 1/y)^m is
    C(m, (m+a+b)/2) * C(m, (m+a-b)/2) for m + a + b even."""
    s = Fraction(0)
    for m in range(abs(a) + abs(b), n + 1):
        if (m + a + b) % 2:
            continue
        s += (math.comb(n, m) * (1 - 4 * alpha) ** (n - m) * alpha ** m
              * math.comb(m, (m + a + b) // 2) * math.comb(m, (m + a - b) // 2))
    return s


def _unaffected_by_edges(nx, ny, ci, cj, n):
    """Cells whose value after n steps equals the unbounded solution: for
    every edge cell e, |e - centre|_1 + |x - e|_1 > n (an edge forced to zero
    at step s can only reach x at step s + |x - e|_1)."""
    ok = np.zeros((ny, nx), dtype=bool)
    edges = [(i, 0) for i in range(nx)] + [(i, ny - 1) for i in range(nx)] + \
            [(0, j) for j in range(ny)] + [(nx - 1, j) for j in range(ny)]
    e = np.array(edges)
    dc = np.abs(e[:, 0] - ci) + np.abs(e[:, 1] - cj)
    for j in range(1, ny - 1):
        for i in range(1, nx - 1):
            dx = np.abs(e[:, 0] - i) + np.abs(e[:, 1] - j)
            ok[j, i] = bool(np.all(dc + dx > n))
    return ok


@pytest.mark.parametrize("nx,ny,n", [(31, 27, 7), (31, 27, 8), (64, 64, 32)])
def test_closed_form_fp64(nx, ny, n):
    """FP64 oracle against the exact closed form on every cell the edges
    cannot reach yet; rounding bound: n steps x ~10 ulps per step."""
    ci, cj = (nx + 1) // 2 - 1, (ny + 1) // 2 - 1
    u = oracle.diffuse2d(oracle.centre_impulse(nx, ny, np.float64), n)
    ok = _unaffected_by_edges(nx, ny, ci, cj, n)
    assert ok.sum() > 100
    tol = n * 10 * 2.0 ** -52
    for j, i in zip(*np.nonzero(ok)):
        exact = _closed_form(i - ci, j - cj, n, ALPHA64)
        if exact == 0:
            assert u[j, i] == 0.0
        else:
            assert abs(Fraction(float(u[j, i])) - exact) <= tol * exact, (i, j)


def test_closed_form_centre_values():
    """The centre after 7 and 8 steps on 31x27 (the edges are 13 cells away)
    and after 32 steps on 64x64 (edges 31 cells away, so the centre is still
    the unbounded value) agrees with the closed form to rounding."""
    for nx, ny, n in ((31, 27, 7), (31, 27, 8), (64, 64, 32)):
        ci, cj = (nx + 1) // 2 - 1, (ny + 1) // 2 - 1
        u = oracle.diffuse2d(oracle.centre_impulse(nx, ny, np.float64), n)
        exact = float(_closed_form(0, 0, n, ALPHA64))
        assert u[cj, ci] == pytest.approx(exact, rel=1e-14, abs=0)


def test_closed_form_fp32():
    """FP32 oracle against the closed form with alpha = the FP32 value of
    0.1; rounding bound n x ~10 FP32 ulps."""
    nx, ny, n = 31, 27, 8
    ci, cj = (nx + 1) // 2 - 1, (ny + 1) // 2 - 1
    u = oracle.diffuse2d(oracle.centre_impulse(nx, ny, np.float32), n)
    ok = _unaffected_by_edges(nx, ny, ci, cj, n)
    tol = n * 10 * 2.0 ** -23
    for j, i in zip(*np.nonzero(ok)):
        exact = _closed_form(i - ci, j - cj, n, ALPHA32)
        got = Fraction(float(u[j, i]))
        assert abs(got - exact) <= tol * exact, (i, j)


# ---------------------------------------------------------------------------
# Exact rational simulation (brute force), edges included
# ---------------------------------------------------------------------------

def _exact_sim(u0: np.ndarray, n: int, alpha: Fraction):
    ny, nx = u0.shape
    u = [[Fraction(float(u0[j, i])) for i in range(nx)] for j in range(ny)]
    for _ in range(n):
        v = [[Fraction(0)] * nx for _ in range(ny)]
        for j in range(1, ny - 1):
            for i in range(1, nx - 1):
                v[j][i] = u[j][i] + alpha * (u[j][i - 1] + u[j][i + 1] + u[j - 1][i]
                                             + u[j + 1][i] - 4 * u[j][i])
        u = v
    return u


@pytest.mark.parametrize("dt,alpha,eps", [(np.float64, ALPHA64, 2.0 ** -52),
                                          (np.float32, ALPHA32, 2.0 ** -23)])
@pytest.mark.parametrize("nx,ny,n", [(9, 7, 5), (12, 10, 11)])
def test_brute_force_random_field(dt, alpha, eps, nx, ny, n):
    """Random interior values, zero edges: the oracle stays within the
    rounding bound n * 8 * eps * max|u0| of the exact rational result at
    every cell, and its edges are exactly zero."""
    u0 = inputs.diffusion_field(nx, ny, dt, seed=inputs.config_seed(0), stream=nx)
    exact = _exact_sim(u0, n, alpha)
    got = oracle.diffuse2d(u0, n)
    bound = n * 8 * eps * float(np.abs(u0).max())
    for j in range(ny):
        for i in range(nx):
            assert abs(Fraction(float(got[j, i])) - exact[j][i]) <= bound, (i, j)
    assert np.all(got[0, :] == 0) and np.all(got[-1, :] == 0)
    assert np.all(got[:, 0] == 0) and np.all(got[:, -1] == 0)


def test_brute_force_nonzero_initial_edges():
    """Initial edges nonzero: each step reads the source edges as they are
    and writes zero to the destination edges (the all-cells loop of the
    Qiita page, section 5.1 and appendix A), so after one step the edges are
    zero and the cells next to them saw the old edge values."""
    nx, ny, n = 10, 8, 3
    u0 = inputs.uniform_f64(inputs.config_seed(0), 99, nx * ny).reshape(ny, nx) + 0.5
    exact = _exact_sim(u0, n, ALPHA64)
    got = oracle.diffuse2d(u0, n)
    for j in range(ny):
        for i in range(nx):
            assert abs(Fraction(float(got[j, i])) - exact[j][i]) <= n * 8 * 2.0 ** -52 * 2, (i, j)
    one = oracle.diffuse2d(u0, 1)
    assert np.all(one[0, :] == 0) and np.all(one[:, -1] == 0)
    assert one[1, 1] == u0[1, 1] + 0.1 * (u0[1, 0] + u0[1, 2] + u0[0, 1] + u0[2, 1] - 4.0 * u0[1, 1])


def test_brute_force_impulse_near_edge():
    """The impulse reaches the edges: 31x27, 16 steps, compared cell by cell
    with the exact rational simulation of the same bounded problem."""
    u0 = oracle.centre_impulse(31, 27, np.float64)
    exact = _exact_sim(u0, 16, ALPHA64)
    got = oracle.diffuse2d(u0, 16)
    for j in range(27):
        for i in range(31):
            e = exact[j][i]
            assert abs(Fraction(float(got[j, i])) - e) <= 16 * 8 * 2.0 ** -52 * max(e, Fraction(1, 10**30))


# ---------------------------------------------------------------------------
# Fronts, symmetry, mass, stability, ping-pong parity
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_axis_front_is_repeated_product(dt):
    """The cell n steps straight out along an axis holds alpha^n, computed
    as n successive rounded products (all other contributions are exact
    zeros), bitwise in both precisions."""
    n = 12
    u = oracle.diffuse2d(oracle.centre_impulse(64, 64, dt), n)
    a = dt(0.1)
    expect = dt(1)
    for _ in range(n):
        expect = dt(a * expect)
    for di, dj in ((n, 0), (-n, 0), (0, n), (0, -n)):
        assert u[31 + dj, 31 + di] == expect


def test_diagonal_front():
    """On the diagonal front |a| + |b| = n the value is C(n, a) alpha^n up to
    rounding."""
    n = 10
    u = oracle.diffuse2d(oracle.centre_impulse(64, 64, np.float64), n)
    for a in range(0, n + 1):
        b = n - a
        exact = math.comb(n, a) * ALPHA64 ** n
        assert abs(Fraction(float(u[31 + b, 31 + a])) - exact) <= 4 * n * 2.0 ** -52 * exact


@pytest.mark.parametrize("n", [7, 8, 31, 32, 60])
def test_i_mirror_bitwise(n):
    """31 columns with the centre in column 15 (0-based): the grid is
    symmetric in i and W+E commutes exactly, so the i-mirror image is
    bitwise identical at every step count."""
    u = oracle.diffuse2d(oracle.centre_impulse(31, 27, np.float64), n)
    assert np.array_equal(u, u[:, ::-1])


def test_j_mirror_and_transpose_to_rounding():
    """Mirroring j swaps S and N and transposing swaps (W,E) with (S,N); the
    left-to-right sum then rounds differently, so these symmetries hold to a
    few ulps only (63x63, centre 31, 40 steps)."""
    u = oracle.diffuse2d(oracle.centre_impulse(63, 63, np.float64), 40)
    scale = float(np.abs(u).max())
    assert np.max(np.abs(u - u[::-1, :])) <= 8 * 2.0 ** -52 * scale
    assert np.max(np.abs(u - u.T)) <= 8 * 2.0 ** -52 * scale
    assert np.array_equal(u, u[:, ::-1])


def test_mass_conserved_until_front_reaches_edge():
    """64x64: the edges are 31 cells from the centre, so the exact mass stays
    1 through step 30 (FP64 within 1e-14)."""
    u = oracle.centre_impulse(64, 64, np.float64)
    for n in range(1, 31):
        u = oracle.diffuse2d(u, 1)
        assert abs(math.fsum(u.ravel().tolist()) - 1.0) <= 1e-14, n


def test_mass_leaks_through_edges_and_never_grows():
    """15x15 (edges 7 cells from the centre): mass is 1 through step 6, then
    leaks through the zero edges and never increases (Qiita appendix A checks
    0 <= mass <= 1 rather than mass = 1 for that reason)."""
    u = oracle.centre_impulse(15, 15, np.float64)
    masses = []
    for n in range(1, 61):
        u = oracle.diffuse2d(u, 1)
        masses.append(math.fsum(u.ravel().tolist()))
        if n <= 6:
            assert abs(masses[-1] - 1.0) <= 1e-15, n
    assert masses[6] < 1.0 - 1e-9
    assert masses[-1] < 0.9
    for a, b in zip(masses, masses[1:]):
        assert b <= a + 1e-15


def test_alpha_quarter_bounded_and_alpha_03_unstable():
    """alpha <= 1/4 makes the update a convex combination: values stay in
    [0, max u0].  alpha = 0.3 amplifies the checkerboard mode by |1 - 8 alpha|
    = 1.4 per step (Qiita section 3 stability condition alpha <= 1/4)."""
    u0 = inputs.diffusion_field(48, 40, np.float64, seed=inputs.config_seed(0), stream=7)
    u = oracle.diffuse2d(u0, 200, alpha=0.25)
    assert u.min() >= 0 and u.max() <= u0.max()
    cb = np.zeros((40, 48))
    jj, ii = np.mgrid[0:40, 0:48]
    cb[1:-1, 1:-1] = (1e-6 * (-1.0) ** (ii + jj))[1:-1, 1:-1]
    grown = oracle.diffuse2d(cb, 100, alpha=0.3)
    assert np.abs(grown).max() > 1e6 * 1e-6
    steady = oracle.diffuse2d(cb, 100, alpha=0.25)
    assert np.abs(steady).max() <= 1e-6


@pytest.mark.parametrize("n", [7, 8, 31, 32])
def test_ping_pong_parity(n):
    """Odd counts leave the result in v and even counts in u; the other
    buffer then holds the previous step (Qiita section 5.4)."""
    for dt in (np.float32, np.float64):
        u0 = oracle.centre_impulse(31, 27, dt)
        u, v, in_v = oracle.diffuse2d(u0, n, return_both=True)
        assert in_v == (n % 2 == 1)
        prev = oracle.diffuse2d(u0, n - 1)
        final = oracle.diffuse2d(u0, n)
        assert np.array_equal(v if in_v else u, final)
        assert np.array_equal(u if in_v else v, prev)


def test_zero_steps_is_identity():
    u0 = inputs.diffusion_field(9, 8, np.float64, seed=1)
    assert np.array_equal(oracle.diffuse2d(u0, 0), u0)


def test_threads_do_not_change_results():
    """The OpenMP build splits the j loop only; results are bitwise those of
    one thread."""
    u0 = inputs.diffusion_field(257, 131, np.float64, seed=inputs.config_seed(2))
    a = oracle.diffuse2d(u0, 9, nthreads=1)
    b = oracle.diffuse2d(u0, 9, nthreads=max(2, oracle.max_threads()))
    assert np.array_equal(a, b)
