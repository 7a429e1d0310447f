"""Seeded synthetic inputs for the field sweeps.

This module is the only code that the GPU path's tests and benchmark share
with the CPU oracle.  It draws numbers and lays them out; it holds none of the
sweeps' arithmetic.  Everything is generated once on the host, in numpy, and
the same host arrays feed both sides.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based hash:
the 64-bit word for element ``n`` of stream ``s`` is
``splitmix64(seed XOR (n + s * 2**40))``, where ``splitmix64(x)`` adds the
golden-gamma constant to ``x`` and applies the published 30/27/31 xor-shift
multiply finaliser.

* uniform FP64 in [0, 1): top 53 bits times 2**-53;
* uniform FP32 in [0, 1): top 24 bits times 2**-24 (exact in FP32);
* standard normal: Box-Muller on consecutive pairs of uniforms
  (u1, u2) -> sqrt(-2 ln(1 - u1)) * (cos, sin)(2 pi u2);
* lognormal: exp of a standard normal (mu = 0, sigma = 1).

Seeds: ``20261202 + config number``; each array of a configuration draws from
its own stream id.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 24


def config_seed(config_number: int) -> int:
    """Seed of the numbered benchmark configuration (1-based)."""
    return SEED_BASE + int(config_number)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def random_bits(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` 64-bit words of stream ``stream``, elements ``start..start+n-1``."""
    out = np.empty(n, dtype=np.uint64)
    key = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    base = np.uint64(start + (int(stream) << 40))
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        ctr = np.arange(lo, hi, dtype=np.uint64) + base
        out[lo:hi] = _splitmix64(ctr ^ key)
    return out


def uniform_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """Uniform FP64 values in [0, 1)."""
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        b = random_bits(seed, stream, hi - lo, lo)
        out[lo:hi] = (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return out


def uniform_f32(seed: int, stream: int, n: int) -> np.ndarray:
    """Uniform FP32 values in [0, 1)."""
    out = np.empty(n, dtype=np.float32)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        b = random_bits(seed, stream, hi - lo, lo)
        out[lo:hi] = ((b >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)).astype(np.float32)
    return out


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """Standard normal FP64 values (Box-Muller on consecutive pairs)."""
    m = (n + 1) // 2
    out = np.empty(2 * m, dtype=np.float64)
    for lo in range(0, m, _CHUNK):
        hi = min(m, lo + _CHUNK)
        u = uniform_f64_range(seed, stream, 2 * lo, 2 * (hi - lo)).reshape(-1, 2)
        r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        th = (2.0 * np.pi) * u[:, 1]
        out[2 * lo:2 * hi:2] = r * np.cos(th)
        out[2 * lo + 1:2 * hi:2] = r * np.sin(th)
    return out[:n]


def uniform_f64_range(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Elements ``start..start+n-1`` of the uniform FP64 stream."""
    b = random_bits(seed, stream, n, start)
    return (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def lognormal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """exp(N(0,1)) values."""
    return np.exp(normal_f64(seed, stream, n))


# ---------------------------------------------------------------------------
# Workload layouts
# ---------------------------------------------------------------------------

def stored_extents(extents, ghost):
    """Stored extents of a field box: n + 2*ghost on axes with n > 1, else 1."""
    return tuple(int(n) + 2 * int(ghost) if int(n) > 1 else 1 for n in extents)


def diffusion_field(nx: int, ny: int, dtype, seed: int | None = None, stream: int = 0,
                    values: str = "uniform"):
    """Initial 2D field of shape (ny, nx) (element [j, i] is u(i, j)).

    With ``seed`` None: the centre impulse (all zero except the 1-based cell
    ((nx+1)/2, (ny+1)/2) = 1).  Otherwise: interior values drawn from the
    seed, edges zero: uniform [0, 1) in the requested precision, or with
    ``values="normal"`` N(0,1) (FP64 draws, rounded to the precision), a
    field of mixed signs.
    """
    dt = np.dtype(dtype)
    u = np.zeros((ny, nx), dtype=dt)
    if seed is None:
        u[(ny + 1) // 2 - 1, (nx + 1) // 2 - 1] = 1
        return u
    n = (nx - 2) * (ny - 2)
    if values == "normal":
        vals = normal_f64(seed, stream, n).astype(dt)
    elif values == "uniform":
        vals = uniform_f32(seed, stream, n) if dt == np.float32 else uniform_f64(seed, stream, n)
    else:
        raise ValueError(f"values must be 'uniform' or 'normal', not {values!r}")
    u[1:-1, 1:-1] = vals.reshape(ny - 2, nx - 2)
    return u


def normal_fields(seed: int, nv: int, extents, ghost: int, first_stream: int = 0):
    """``nv`` stored boxes of N(0,1) values, each a flat FP64 array in
    Fortran order (element (j,k,l) at j + N1*(k + N2*l))."""
    n = int(np.prod(stored_extents(extents, ghost)))
    return [normal_f64(seed, first_stream + i, n) for i in range(nv)]


def face_fluxes(seed: int, nv: int, extents, direction: int, stream: int = 100):
    """Face-flux array ~ N(0,1) with one more entry along ``direction``;
    flat FP64, variable index slowest."""
    e = [int(x) for x in extents]
    e[direction] += 1
    return normal_f64(seed, stream + direction, int(np.prod(e)) * nv)


def inverse_spacing(seed: int, n: int, stream: int = 200):
    """inv_d = 1/d with d ~ U[0.5, 1.5]/n, computed on the host once."""
    d = (0.5 + uniform_f64(seed, stream, n)) / n
    return 1.0 / d


def multivar_fields_2d(seed: int, extents, ghost: int):
    """The seven fields of the 2D multi-variable sweep (2 partial densities,
    2 momenta, energy, 2 volume fractions): densities and energy lognormal,
    momenta N(0,1), volume fractions uniform [0, 1).  Ghost cells are drawn
    like interior cells."""
    n = int(np.prod(stored_extents(extents, ghost)))
    return [
        lognormal_f64(seed, 0, n),  # partial density 1
        lognormal_f64(seed, 1, n),  # partial density 2
        normal_f64(seed, 2, n),     # momentum x
        normal_f64(seed, 3, n),     # momentum y
        lognormal_f64(seed, 4, n),  # energy
        uniform_f64(seed, 5, n),    # volume fraction 1
        uniform_f64(seed, 6, n),    # volume fraction 2
    ]
