"""CPU oracle for the per-cell field sweeps -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never imports it and it
never imports the GPU library; the only code the two sides share is the seeded
input generator module, which holds none of the method's arithmetic.

The arithmetic lives in ``fvf_oracle.c`` (plain C, built with
``-O2 -ffp-contract=off``); this module loads it with ctypes, wraps it for
numpy arrays and adds the comparison metrics and physical checks that the
Qiita page ("Fortran 2018 GPU acceleration, part 3") describes in its
section 8 (tolerance model, section 8.1 metrics) and in its appendix A
(``print_summary``: finiteness, bounds and mass checks).

Parity status of every function here: pinned (see tests/test_oracle_*.py).
"""
from __future__ import annotations

import ctypes
import math
import os
import shutil
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "fvf_oracle.c"
_LIB = _HERE / "liboracle_fvf.so"
_lib = None

# Flags: no FMA contraction (every multiply and add rounded on its own), no
# -march=native (the same results on x86-64 and aarch64 hosts).
_CFLAGS = ["-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> Path:
    """Compile ``fvf_oracle.c`` into ``liboracle_fvf.so`` (with OpenMP if gcc
    supports it).  Does nothing when the library is newer than the source."""
    if (not force and _LIB.exists()
            and _LIB.stat().st_mtime >= _SRC.stat().st_mtime):
        return _LIB
    cc = os.environ.get("CC") or shutil.which("gcc") or "cc"
    tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
    base = [cc, *_CFLAGS, str(_SRC), "-o", str(tmp)]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(str(_LIB))
    i64, dbl, flt, cint = ctypes.c_int64, ctypes.c_double, ctypes.c_float, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_diffuse2d_f64.argtypes = [vp, vp, i64, i64, dbl, i64, cint]
    lib.oracle_diffuse2d_f64.restype = cint
    lib.oracle_diffuse2d_f32.argtypes = [vp, vp, i64, i64, flt, i64, cint]
    lib.oracle_diffuse2d_f32.restype = cint
    lib.oracle_diffuse3d_f64.argtypes = [vp, vp, i64, i64, i64, dbl, i64, cint]
    lib.oracle_diffuse3d_f64.restype = cint
    lib.oracle_diffuse3d_f32.argtypes = [vp, vp, i64, i64, i64, flt, i64, cint]
    lib.oracle_diffuse3d_f32.restype = cint
    lib.oracle_weno_pack.argtypes = [ctypes.POINTER(vp), cint, i64, i64, i64, i64, cint, vp]
    lib.oracle_weno_pack.restype = cint
    lib.oracle_advect_rhs.argtypes = [vp, vp, cint, i64, i64, i64, cint, vp]
    lib.oracle_advect_rhs.restype = cint
    lib.oracle_advect_rhs_add.argtypes = [vp, vp, cint, i64, i64, i64, cint, vp]
    lib.oracle_advect_rhs_add.restype = cint
    lib.oracle_flux_unpack.argtypes = [vp, cint, i64, i64, i64, cint, vp]
    lib.oracle_flux_unpack.restype = cint
    lib.oracle_fields_copy.argtypes = [ctypes.POINTER(vp), cint, i64, i64, i64, i64,
                                       ctypes.POINTER(vp)]
    lib.oracle_fields_copy.restype = cint
    lib.oracle_rk_axpby.argtypes = [vp, vp, vp, i64, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, vp]
    lib.oracle_rk_axpby.restype = cint
    lib.oracle_weno_pack_f32.argtypes = [ctypes.POINTER(vp), cint, i64, i64, i64, i64, cint, vp]
    lib.oracle_weno_pack_f32.restype = cint
    lib.oracle_advect_rhs_f32.argtypes = [vp, vp, cint, i64, i64, i64, cint, cint, vp]
    lib.oracle_advect_rhs_f32.restype = cint
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = cint
    _lib = lib
    return lib


def max_threads() -> int:
    """Threads the OpenMP build may use (1 if built without OpenMP)."""
    return int(_load().oracle_max_threads())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---------------------------------------------------------------------------
# 2D diffusion
# ---------------------------------------------------------------------------

def diffuse2d(u0: np.ndarray, nsteps: int, alpha: float = 0.1, v0: np.ndarray | None = None,
              nthreads: int = 1, return_both: bool = False):
    """Run ``nsteps`` ping-pong applications of the 5-point update.

    ``u0`` is the initial field as a numpy array of shape (ny, nx) in C order,
    i.e. element [j, i] is u(i, j) at address i + nx*j -- the column-major
    Fortran layout of the Qiita page (section 4).  ``v0`` is the initial second
    buffer (zeros if None).  The dtype (float32 or float64) selects the
    precision; for float32 ``alpha`` is rounded once to FP32.

    Returns the final field (copy), or (u, v, result_in_v) if ``return_both``.
    """
    u = np.array(u0, copy=True, order="C")
    if u.ndim != 2:
        raise ValueError("u0 must be 2D (ny, nx)")
    ny, nx = u.shape
    v = np.zeros_like(u) if v0 is None else np.array(v0, dtype=u.dtype, copy=True, order="C")
    lib = _load()
    if u.dtype == np.float64:
        in_v = lib.oracle_diffuse2d_f64(_ptr(u), _ptr(v), nx, ny, float(alpha), int(nsteps),
                                        int(nthreads))
    elif u.dtype == np.float32:
        in_v = lib.oracle_diffuse2d_f32(_ptr(u), _ptr(v), nx, ny,
                                        float(np.float32(alpha)), int(nsteps), int(nthreads))
    else:
        raise TypeError("dtype must be float32 or float64")
    if return_both:
        return u, v, bool(in_v)
    return v if in_v else u


def diffuse3d(u0: np.ndarray, nsteps: int, alpha: float = 0.1, v0: np.ndarray | None = None,
              nthreads: int = 1, return_both: bool = False):
    """``nsteps`` ping-pong applications of the 7-point update on a 3D grid.

    ``u0`` has shape (nz, ny, nx) in C order: element [k, j, i] is u(i, j, k)
    at address i + nx*(j + ny*k), the column-major layout with i fastest.
    Otherwise as ``diffuse2d``.
    """
    u = np.array(u0, copy=True, order="C")
    if u.ndim != 3:
        raise ValueError("u0 must be 3D (nz, ny, nx)")
    nz, ny, nx = u.shape
    v = np.zeros_like(u) if v0 is None else np.array(v0, dtype=u.dtype, copy=True, order="C")
    lib = _load()
    if u.dtype == np.float64:
        in_v = lib.oracle_diffuse3d_f64(_ptr(u), _ptr(v), nx, ny, nz, float(alpha), int(nsteps),
                                        int(nthreads))
    elif u.dtype == np.float32:
        in_v = lib.oracle_diffuse3d_f32(_ptr(u), _ptr(v), nx, ny, nz,
                                        float(np.float32(alpha)), int(nsteps), int(nthreads))
    else:
        raise TypeError("dtype must be float32 or float64")
    if return_both:
        return u, v, bool(in_v)
    return v if in_v else u


def centre_impulse(nx: int, ny: int, dtype=np.float64) -> np.ndarray:
    """Initial field of the Qiita page (appendix A, set_initial_condition):
    all zero except the cell ((nx+1)/2, (ny+1)/2) (1-based, integer division)
    which is 1.  Returned as shape (ny, nx)."""
    u = np.zeros((ny, nx), dtype=dtype)
    u[(ny + 1) // 2 - 1, (nx + 1) // 2 - 1] = 1
    return u


# ---------------------------------------------------------------------------
# 3D box sweeps
# ---------------------------------------------------------------------------

def stored_extents(extents, ghost):
    """Stored extents (N1, N2, N3): n + 2g on axes with n > 1, else 1."""
    return tuple(n + 2 * ghost if n > 1 else 1 for n in extents)


def pack_extents(extents, ghost, direction):
    """Output extents (M1, M2, M3) of the pack for direction 0/1/2."""
    n1, n2, n3 = extents
    N1, N2, N3 = stored_extents(extents, ghost)
    return [(N1, n2, n3), (N2, n1, n3), (N3, n2, n1)][direction]


def flux_extents(extents, direction):
    """Extents (F1, F2, F3) of the face-flux array for direction 0/1/2."""
    e = list(extents)
    e[direction] += 1
    return tuple(e)


def weno_pack(fields, extents, ghost: int, direction: int) -> np.ndarray:
    """The WENO input pack (MFC pull request #2087, "Changes").

    ``fields`` is a list of nv arrays, all float64 or all float32 (the FP32
    form, a 4-byte copy), each holding the stored box in Fortran order
    (element (j,k,l) at j + N1*(k + N2*l)); any shape with that many elements
    is accepted, other dtypes are converted to float64.  Returns a flat array
    of M1*M2*M3*nv elements of the fields' dtype, laid out as described in
    ``fvf_oracle.c``.
    """
    n1, n2, n3 = (int(x) for x in extents)
    nst = int(np.prod(stored_extents(extents, ghost)))
    f32 = len(fields) > 0 and all(np.asarray(f).dtype == np.float32 for f in fields)
    dt = np.float32 if f32 else np.float64
    arrs = []
    for f in fields:
        a = np.ascontiguousarray(f, dtype=dt).reshape(-1)
        if a.size != nst:
            raise ValueError(f"field has {a.size} elements, expected {nst}")
        arrs.append(a)
    nv = len(arrs)
    out = np.empty(int(np.prod(pack_extents(extents, ghost, direction))) * nv, dtype=dt)
    table = (ctypes.c_void_p * max(1, nv))(*[_ptr(a) for a in arrs])
    fn = _load().oracle_weno_pack_f32 if f32 else _load().oracle_weno_pack
    rc = fn(table, nv, n1, n2, n3, int(ghost), int(direction), _ptr(out))
    if rc != 0:
        raise ValueError("bad direction")
    return out


def _flux_args(flux, inv_d, nv, extents, direction):
    n1, n2, n3 = (int(x) for x in extents)
    f32 = np.asarray(flux).dtype == np.float32
    dt = np.float32 if f32 else np.float64
    fl = np.ascontiguousarray(flux, dtype=dt).reshape(-1)
    w = np.ascontiguousarray(inv_d, dtype=dt).reshape(-1)
    if fl.size != int(np.prod(flux_extents(extents, direction))) * nv:
        raise ValueError("flux size mismatch")
    if w.size != (n1, n2, n3)[direction]:
        raise ValueError("inv_d size mismatch")
    return n1, n2, n3, f32, dt, fl, w


def advect_rhs(flux: np.ndarray, inv_d: np.ndarray, nv: int, extents, direction: int) -> np.ndarray:
    """The flux-difference source (MFC pull request #2087, "Changes",
    s_compute_advection_source_term); layout as in ``fvf_oracle.c``.  A
    float32 flux selects the FP32 form (inv_d converted to float32)."""
    n1, n2, n3, f32, dt, fl, w = _flux_args(flux, inv_d, nv, extents, direction)
    rhs = np.empty(n1 * n2 * n3 * nv, dtype=dt)
    if f32:
        rc = _load().oracle_advect_rhs_f32(_ptr(fl), _ptr(w), int(nv), n1, n2, n3,
                                           int(direction), 0, _ptr(rhs))
    else:
        rc = _load().oracle_advect_rhs(_ptr(fl), _ptr(w), int(nv), n1, n2, n3, int(direction),
                                       _ptr(rhs))
    if rc != 0:
        raise ValueError("bad direction")
    return rhs


def advect_rhs_add(flux: np.ndarray, inv_d: np.ndarray, nv: int, extents, direction: int,
                   rhs: np.ndarray) -> np.ndarray:
    """rhs + the flux-difference term of ``direction`` (returns a new array):
    the accumulating form that builds the finite-volume right-hand side over
    the directions.  A float32 flux selects the FP32 form."""
    n1, n2, n3, f32, dt, fl, w = _flux_args(flux, inv_d, nv, extents, direction)
    out = np.array(rhs, dtype=dt, copy=True).reshape(-1)
    if out.size != n1 * n2 * n3 * nv:
        raise ValueError("size mismatch")
    if f32:
        rc = _load().oracle_advect_rhs_f32(_ptr(fl), _ptr(w), int(nv), n1, n2, n3,
                                           int(direction), 1, _ptr(out))
    else:
        rc = _load().oracle_advect_rhs_add(_ptr(fl), _ptr(w), int(nv), n1, n2, n3,
                                           int(direction), _ptr(out))
    if rc != 0:
        raise ValueError("bad direction")
    return out


def sweep_flux_extents(extents, direction):
    """Extents of a sweep-frame face array (swept axis first, n+1 faces)."""
    n1, n2, n3 = (int(x) for x in extents)
    return [(n1 + 1, n2, n3), (n2 + 1, n1, n3), (n3 + 1, n2, n1)][direction]


def flux_unpack(sweep_flux: np.ndarray, nv: int, extents, direction: int) -> np.ndarray:
    """Directional flux copy from the sweep frame to the physical frame
    (MFC pull request #2087, "Changes", s_finalize_riemann_solver); layout
    as in ``fvf_oracle.c``."""
    n1, n2, n3 = (int(x) for x in extents)
    src = np.ascontiguousarray(sweep_flux, dtype=np.float64).reshape(-1)
    size = int(np.prod(flux_extents(extents, direction))) * nv
    if src.size != size:
        raise ValueError("size mismatch")
    out = np.empty(size, dtype=np.float64)
    rc = _load().oracle_flux_unpack(_ptr(src), int(nv), n1, n2, n3, int(direction), _ptr(out))
    if rc != 0:
        raise ValueError("bad direction")
    return out


def fields_copy(fields, extents, ghost: int):
    """The conservative-variable copy (MFC pull request #2087, "Changes",
    s_compute_rhs): a new array per field holding its whole stored box."""
    n1, n2, n3 = (int(x) for x in extents)
    nst = int(np.prod(stored_extents(extents, ghost)))
    src = [np.ascontiguousarray(f, dtype=np.float64).reshape(-1) for f in fields]
    if any(a.size != nst for a in src):
        raise ValueError("field size mismatch")
    dst = [np.empty(nst, dtype=np.float64) for _ in src]
    st = (ctypes.c_void_p * max(1, len(src)))(*[_ptr(a) for a in src])
    dt = (ctypes.c_void_p * max(1, len(dst)))(*[_ptr(a) for a in dst])
    _load().oracle_fields_copy(st, len(src), n1, n2, n3, int(ghost), dt)
    return dst


def weno_pack_copy(fields, extents, ghost: int, direction: int):
    """The pack fused with the conservative-variable copy: (packed, copies),
    the two results of one pass over the fields."""
    return weno_pack(fields, extents, ghost, direction), fields_copy(fields, extents, ghost)


# Shu-Osher SSPRK3 stage coefficients (a, b) of out = a*u^n + b*(u + dt*rhs).
SSPRK3_STAGES = ((0.0, 1.0), (0.75, 0.25), (1.0 / 3.0, 2.0 / 3.0))


def rk_axpby(u0, u, rhs, a: float, b: float, dt: float):
    """One SSPRK3 stage update out = a*u0 + b*(u + dt*rhs) (Mallard
    documentation, "Design: single-GPU performance and parallel scaling",
    "Baseline (main)": axpby per stage)."""
    u0 = np.ascontiguousarray(u0, dtype=np.float64).reshape(-1)
    u = np.ascontiguousarray(u, dtype=np.float64).reshape(-1)
    rhs = np.ascontiguousarray(rhs, dtype=np.float64).reshape(-1)
    if not (u0.size == u.size == rhs.size):
        raise ValueError("size mismatch")
    out = np.empty_like(u)
    _load().oracle_rk_axpby(_ptr(u0), _ptr(u), _ptr(rhs), u.size, float(a), float(b), float(dt),
                            _ptr(out))
    return out


def fv_rhs(fluxes, inv_ds, nv: int, extents):
    """The finite-volume right-hand side from face fluxes: the x difference
    assigned, then the y and z differences added in that order (a direction
    whose flux is None is skipped; x must be given)."""
    if fluxes[0] is None:
        raise ValueError("the x flux is required")
    rhs = advect_rhs(fluxes[0], inv_ds[0], nv, extents, 0)
    for d in (1, 2):
        if fluxes[d] is not None:
            rhs = advect_rhs_add(fluxes[d], inv_ds[d], nv, extents, d, rhs)
    return rhs


def ssprk3_stage(u0, u, fluxes, inv_ds, nv: int, extents, a: float, b: float, dt: float):
    """The stage update fused with the flux difference: rhs from the face
    fluxes (fv_rhs), then out = a*u0 + b*(u + dt*rhs)."""
    return rk_axpby(u0, u, fv_rhs(fluxes, inv_ds, nv, extents), a, b, dt)


def multivar_sweep_2d(fields, fluxes_x, fluxes_y, inv_dx, inv_dy, nv, extents, ghost):
    """One repetition of the 2D multi-variable sequence: pack x, pack y,
    flux difference x, flux difference y (each an assignment; the y pass
    overwrites the rhs of the x pass).  Returns (packed_x, packed_y, rhs_x,
    rhs_y) so that every output of the sequence can be compared."""
    px = weno_pack(fields, extents, ghost, 0)
    py = weno_pack(fields, extents, ghost, 1)
    rx = advect_rhs(fluxes_x, inv_dx, nv, extents, 0)
    ry = advect_rhs(fluxes_y, inv_dy, nv, extents, 1)
    return px, py, rx, ry


# ---------------------------------------------------------------------------
# Comparison metrics and physical checks (Qiita section 8, appendix A)
# ---------------------------------------------------------------------------

def compare_fields(reference: np.ndarray, candidate: np.ndarray, atol: float, rtol: float) -> dict:
    """Whole-grid comparison of a candidate against a reference field.

    Both are converted exactly to float64.  A cell fails when
    |ref - cand| > atol + rtol*|ref| (Qiita section 8).  Reports, as the
    page's section 8.1 lists them: the largest absolute difference and where
    it is (0-based flat index), the root-mean-square difference, the relative
    L2 difference (difference norm over reference norm), the mass difference
    (sum of candidate minus sum of reference, each summed exactly with
    math.fsum), the number of failing cells and the number of cells.
    """
    ref = np.asarray(reference, dtype=np.float64).reshape(-1)
    cand = np.asarray(candidate, dtype=np.float64).reshape(-1)
    if ref.shape != cand.shape:
        raise ValueError("shape mismatch")
    d = np.abs(ref - cand)
    dl = d.tolist()
    rl = ref.tolist()
    sq_err = math.fsum(x * x for x in dl)
    sq_ref = math.fsum(x * x for x in rl)
    worst = int(np.argmax(d))
    return {
        "max_abs": float(d[worst]),
        "worst_index": worst,
        "rmse": math.sqrt(sq_err / len(dl)),
        "relative_l2": math.sqrt(sq_err / sq_ref) if sq_ref else math.sqrt(sq_err),
        "mass_difference": math.fsum(cand.tolist()) - math.fsum(rl),
        "failures": int(np.count_nonzero(d > atol + rtol * np.abs(ref))),
        "cells": len(dl),
    }


def physical_check(field: np.ndarray) -> dict:
    """The checks the Qiita page's programs run on every result (appendix A,
    print_summary): all values finite, min >= -tol, max <= 1 + tol and
    -tol <= mass <= 1 + tol, with tol = 1e-4 for FP32 and 1e-10 for FP64.
    Returns the quantities and a boolean ``ok``."""
    f = np.asarray(field)
    tol = 1e-4 if f.dtype == np.float32 else 1e-10
    f64 = f.astype(np.float64)
    mass = float(np.sum(f64))
    mn, mx = float(f64.min()), float(f64.max())
    ok = bool(np.all(np.isfinite(f64))) and mn >= -tol and mx <= 1.0 + tol \
        and -tol <= mass <= 1.0 + tol
    return {"ok": ok, "mass": mass, "min": mn, "max": mx, "tol": tol}
