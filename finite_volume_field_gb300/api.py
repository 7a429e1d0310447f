"""Python binding of libfvf.so (include/fvf.h): argument marshalling only.

Every function here converts its arguments to the C ABI's plain pointers and
sizes, calls the library and raises ``FvfError`` on a nonzero status.  All
arithmetic runs in the library's CUDA kernels; there is no other code path.
If the library is missing the first call raises, it never falls back.

Array arguments are torch CUDA tensors (contiguous, of the stated dtype) or
plain integers holding device addresses.  ``stream`` is a torch.cuda.Stream,
a raw cudaStream_t integer, or None for torch's current stream.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libfvf.so"

FVF_FP32 = 0
FVF_FP64 = 1
MAX_NV = 64

_lib = None


class FvfError(RuntimeError):
    """A nonzero status from libfvf."""

    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func}: status {status} ({message})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libfvf.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(
            f"libfvf.so not found at {LIB_PATH}; build it with "
            "`python -m finite_volume_field_gb300.buildlib` (needs nvcc)")
    lib = ctypes.CDLL(str(LIB_PATH))
    i64, vp, cint = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.diffuse2d_step.argtypes = [vp, vp, i64, i64, ctypes.c_double, i64, cint, vp]
    lib.diffuse2d_step.restype = cint
    lib.diffuse3d_step.argtypes = [vp, vp, i64, i64, i64, ctypes.c_double, i64, cint, vp]
    lib.diffuse3d_step.restype = cint
    lib.weno_pack.argtypes = [ctypes.POINTER(vp), cint, ctypes.POINTER(i64), cint, cint, vp, vp]
    lib.weno_pack.restype = cint
    lib.weno_pack_f32.argtypes = [ctypes.POINTER(vp), cint, ctypes.POINTER(i64), cint, cint, vp,
                                  vp]
    lib.weno_pack_f32.restype = cint
    for name in ("advect_rhs_f32", "advect_rhs_add_f32"):
        getattr(lib, name).argtypes = [vp, vp, cint, ctypes.POINTER(i64), cint, vp, vp]
        getattr(lib, name).restype = cint
    lib.advect_rhs.argtypes = [vp, vp, cint, ctypes.POINTER(i64), cint, vp, vp]
    lib.advect_rhs.restype = cint
    lib.advect_rhs_add.argtypes = [vp, vp, cint, ctypes.POINTER(i64), cint, vp, vp]
    lib.advect_rhs_add.restype = cint
    lib.flux_unpack.argtypes = [vp, cint, ctypes.POINTER(i64), cint, vp, vp]
    lib.flux_unpack.restype = cint
    lib.fields_copy.argtypes = [ctypes.POINTER(vp), cint, ctypes.POINTER(i64), cint,
                                ctypes.POINTER(vp), vp]
    lib.fields_copy.restype = cint
    lib.weno_pack_copy.argtypes = [ctypes.POINTER(vp), cint, ctypes.POINTER(i64), cint, cint, vp,
                                   ctypes.POINTER(vp), vp]
    lib.weno_pack_copy.restype = cint
    dbl = ctypes.c_double
    lib.ssprk3_axpby.argtypes = [vp, vp, vp, cint, ctypes.POINTER(i64), dbl, dbl, dbl, vp, vp]
    lib.ssprk3_axpby.restype = cint
    lib.ssprk3_stage.argtypes = [vp, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), cint,
                                 ctypes.POINTER(i64), dbl, dbl, dbl, vp, vp]
    lib.ssprk3_stage.restype = cint
    lib.fvf_status_string.argtypes = [cint]
    lib.fvf_status_string.restype = ctypes.c_char_p
    lib.fvf_last_cuda_error.argtypes = []
    lib.fvf_last_cuda_error.restype = cint
    lib.fvf_device_error.argtypes = [ctypes.POINTER(cint)]
    lib.fvf_device_error.restype = cint
    lib.fvf_launch_count.argtypes = []
    lib.fvf_launch_count.restype = ctypes.c_uint64
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fvf_status_string(int(status)).decode()


def launch_count() -> int:
    """Kernels launched by the library since it was loaded."""
    return int(load().fvf_launch_count())


def device_error() -> int:
    """Reads and clears the device error flags: bit 1, a kernel's bounded
    wait on its own copies expired; bit 2 (index-checking builds), a kernel
    met an out-of-range index.  0: none.  Synchronises the device."""
    flag = ctypes.c_int(0)
    _check("fvf_device_error", load().fvf_device_error(ctypes.byref(flag)))
    return int(flag.value)


def last_cuda_error() -> int:
    return int(load().fvf_last_cuda_error())


def _check(func: str, status: int):
    if status != 0:
        msg = status_string(status)
        if status == 11:
            msg += f" (cudaError {last_cuda_error()})"
        raise FvfError(func, status, msg)


def _addr(x, dtype=None, name="array"):
    """Device address of a torch CUDA tensor (checked) or an int address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch  # deferred: the binding needs torch only for tensors
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or an int address")
    if not x.is_cuda:
        raise ValueError(f"{name}: tensor must be on a CUDA device")
    if not x.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {x.dtype}")
    return x.data_ptr() if x.numel() else None


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _extents(extents):
    e = [int(x) for x in extents]
    if len(e) != 3:
        raise ValueError("extents must have three entries (n1, n2, n3)")
    return (ctypes.c_int64 * 3)(*e)


def diffuse2d_step(u, v, nx: int, ny: int, alpha: float, nsteps: int, dtype: int | None = None,
                   stream=None) -> None:
    """Enqueue ``nsteps`` ping-pong 5-point diffusion steps (include/fvf.h).

    ``dtype`` is FVF_FP32 / FVF_FP64; if None it is taken from ``u``'s torch
    dtype.  The result is in ``v`` after an odd count, in ``u`` after an even
    one.
    """
    if dtype is None:
        import torch
        dtype = FVF_FP64 if u.dtype == torch.float64 else FVF_FP32
    tdt = None
    if not isinstance(u, int):
        import torch
        tdt = torch.float64 if dtype == FVF_FP64 else torch.float32
    st = load().diffuse2d_step(_addr(u, tdt, "u"), _addr(v, tdt, "v"), int(nx), int(ny),
                               float(alpha), int(nsteps), int(dtype), _stream(stream))
    _check("diffuse2d_step", st)


def diffuse3d_step(u, v, nx: int, ny: int, nz: int, alpha: float, nsteps: int,
                   dtype: int | None = None, stream=None) -> None:
    """Enqueue ``nsteps`` ping-pong 7-point diffusion steps on an nx*ny*nz
    grid (include/fvf.h); dtype as for ``diffuse2d_step``."""
    if dtype is None:
        import torch
        dtype = FVF_FP64 if u.dtype == torch.float64 else FVF_FP32
    tdt = None
    if not isinstance(u, int):
        import torch
        tdt = torch.float64 if dtype == FVF_FP64 else torch.float32
    st = load().diffuse3d_step(_addr(u, tdt, "u"), _addr(v, tdt, "v"), int(nx), int(ny), int(nz),
                               float(alpha), int(nsteps), int(dtype), _stream(stream))
    _check("diffuse3d_step", st)


def weno_pack(fields, nv: int, extents, ghost: int, dir: int, out, stream=None) -> None:
    """Enqueue the WENO input pack of ``nv`` fields along ``dir``."""
    import torch
    ptrs = [_addr(f, torch.float64, f"fields[{i}]") for i, f in enumerate(list(fields)[:nv])]
    table = (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)
    st = load().weno_pack(table if ptrs else None, int(nv), _extents(extents), int(ghost),
                          int(dir), _addr(out, torch.float64, "out"), _stream(stream))
    _check("weno_pack", st)


def weno_pack_f32(fields, nv: int, extents, ghost: int, dir: int, out, stream=None) -> None:
    """Enqueue the WENO input pack of ``nv`` FP32 fields along ``dir``."""
    import torch
    ptrs = [_addr(f, torch.float32, f"fields[{i}]") for i, f in enumerate(list(fields)[:nv])]
    table = (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)
    st = load().weno_pack_f32(table if ptrs else None, int(nv), _extents(extents), int(ghost),
                              int(dir), _addr(out, torch.float32, "out"), _stream(stream))
    _check("weno_pack_f32", st)


def advect_rhs_f32(flux, inv_d, nv: int, extents, dir: int, rhs, stream=None) -> None:
    """Enqueue the FP32 flux-difference source along ``dir``."""
    import torch
    f32 = torch.float32
    st = load().advect_rhs_f32(_addr(flux, f32, "flux"), _addr(inv_d, f32, "inv_d"), int(nv),
                               _extents(extents), int(dir), _addr(rhs, f32, "rhs"),
                               _stream(stream))
    _check("advect_rhs_f32", st)


def advect_rhs_add_f32(flux, inv_d, nv: int, extents, dir: int, rhs, stream=None) -> None:
    """Enqueue rhs += the FP32 flux-difference term along ``dir``."""
    import torch
    f32 = torch.float32
    st = load().advect_rhs_add_f32(_addr(flux, f32, "flux"), _addr(inv_d, f32, "inv_d"), int(nv),
                                   _extents(extents), int(dir), _addr(rhs, f32, "rhs"),
                                   _stream(stream))
    _check("advect_rhs_add_f32", st)


def advect_rhs(flux, inv_d, nv: int, extents, dir: int, rhs, stream=None) -> None:
    """Enqueue the flux-difference source along ``dir``."""
    import torch
    st = load().advect_rhs(_addr(flux, torch.float64, "flux"), _addr(inv_d, torch.float64, "inv_d"),
                           int(nv), _extents(extents), int(dir), _addr(rhs, torch.float64, "rhs"),
                           _stream(stream))
    _check("advect_rhs", st)


def advect_rhs_add(flux, inv_d, nv: int, extents, dir: int, rhs, stream=None) -> None:
    """Enqueue rhs += the flux-difference term along ``dir``."""
    import torch
    st = load().advect_rhs_add(_addr(flux, torch.float64, "flux"),
                               _addr(inv_d, torch.float64, "inv_d"), int(nv), _extents(extents),
                               int(dir), _addr(rhs, torch.float64, "rhs"), _stream(stream))
    _check("advect_rhs_add", st)


def flux_unpack(sweep_flux, nv: int, extents, dir: int, out, stream=None) -> None:
    """Enqueue the directional flux copy from the sweep frame to the physical
    frame."""
    import torch
    st = load().flux_unpack(_addr(sweep_flux, torch.float64, "sweep_flux"), int(nv),
                            _extents(extents), int(dir), _addr(out, torch.float64, "out"),
                            _stream(stream))
    _check("flux_unpack", st)


def _table(arrays, nv: int, name: str):
    import torch
    ptrs = [_addr(a, torch.float64, f"{name}[{i}]") for i, a in enumerate(list(arrays)[:nv])]
    return (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs) if ptrs else None


def fields_copy(fields, nv: int, extents, ghost: int, copies, stream=None) -> None:
    """Enqueue the conservative-variable copy copies[i] = fields[i]."""
    st = load().fields_copy(_table(fields, nv, "fields"), int(nv), _extents(extents), int(ghost),
                            _table(copies, nv, "copies"), _stream(stream))
    _check("fields_copy", st)


def weno_pack_copy(fields, nv: int, extents, ghost: int, dir: int, out, copies,
                   stream=None) -> None:
    """Enqueue the WENO input pack along ``dir`` fused with the
    conservative-variable copy of the same fields."""
    import torch
    st = load().weno_pack_copy(_table(fields, nv, "fields"), int(nv), _extents(extents),
                               int(ghost), int(dir), _addr(out, torch.float64, "out"),
                               _table(copies, nv, "copies"), _stream(stream))
    _check("weno_pack_copy", st)


def ssprk3_axpby(u0, u, rhs, nv: int, extents, a: float, b: float, dt: float, out,
                 stream=None) -> None:
    """Enqueue one SSPRK3 stage update out = a*u0 + b*(u + dt*rhs)."""
    import torch
    f64 = torch.float64
    st = load().ssprk3_axpby(_addr(u0, f64, "u0"), _addr(u, f64, "u"), _addr(rhs, f64, "rhs"),
                             int(nv), _extents(extents), float(a), float(b), float(dt),
                             _addr(out, f64, "out"), _stream(stream))
    _check("ssprk3_axpby", st)


def ssprk3_stage(u0, u, fluxes, inv_ds, nv: int, extents, a: float, b: float, dt: float, out,
                 stream=None) -> None:
    """Enqueue the SSPRK3 stage update fused with the flux difference;
    ``fluxes`` and ``inv_ds`` are three entries each (x, y, z), y and z may be
    None."""
    import torch
    f64 = torch.float64
    fl = [_addr(f, f64, f"fluxes[{d}]") for d, f in enumerate(list(fluxes)[:3])]
    w = [_addr(x, f64, f"inv_ds[{d}]") if x is not None else None
         for d, x in enumerate(list(inv_ds)[:3])]
    fl += [None] * (3 - len(fl))
    w += [None] * (3 - len(w))
    st = load().ssprk3_stage(_addr(u0, f64, "u0"), _addr(u, f64, "u"), (ctypes.c_void_p * 3)(*fl),
                             (ctypes.c_void_p * 3)(*w), int(nv), _extents(extents), float(a),
                             float(b), float(dt), _addr(out, f64, "out"), _stream(stream))
    _check("ssprk3_stage", st)
