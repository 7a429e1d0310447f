"""Host-side checks of the C ABI (no GPU needed).

libfvf.so must load, export exactly the functions include/fvf.h declares,
and reject bad arguments with the documented status codes before anything
reaches the GPU.  No call here launches a kernel.
"""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import numpy as np
import pytest

from finite_volume_field_gb300 import api, buildlib

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "fvf.h"


@pytest.fixture(scope="module")
def lib():
    buildlib.build()
    return api.load()


def _declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M))


def _status_codes():
    return {m.group(1): int(m.group(2))
            for m in re.finditer(r"#define\s+(FVF_\w+)\s+(-?\d+)", HEADER.read_text())}


def test_header_declares_the_three_sweeps():
    decl = _declared_functions()
    assert {"diffuse2d_step", "weno_pack", "advect_rhs", "fvf_status_string"} <= decl


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(api.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    exported = {s for s in exported if not s.startswith("_")}
    assert exported == _declared_functions()


def test_status_strings(lib):
    codes = _status_codes()
    seen = set()
    for name, code in codes.items():
        if name.startswith("FVF_ERR_") or name == "FVF_OK":
            s = api.status_string(code)
            assert s != "unknown status"
            seen.add(s)
    assert api.status_string(12345) == "unknown status"
    assert len(seen) == sum(1 for n in codes if n.startswith("FVF_ERR_") or n == "FVF_OK")


C = _status_codes()
E3 = (ctypes.c_int64 * 3)


def test_diffuse_validation(lib):
    f = lib.diffuse2d_step
    assert f(None, None, 8, 8, 0.1, 1, 2, None) == C["FVF_ERR_DTYPE"]
    assert f(None, None, -1, 8, 0.1, 1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(None, None, 8, 8, 0.1, -1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(None, None, 1 << 40, 1 << 40, 0.1, 1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(None, None, 8, 8, float("inf"), 1, 1, None) == C["FVF_ERR_ALPHA"]
    assert f(None, None, 8, 8, float("nan"), 1, 0, None) == C["FVF_ERR_ALPHA"]
    assert f(None, None, 8, 8, 1e300, 1, 0, None) == C["FVF_ERR_ALPHA"]   # inf once rounded to FP32
    assert f(None, None, 8, 8, 0.1, 0, 1, None) == C["FVF_OK"]            # nothing to do
    assert f(None, None, 0, 8, 0.1, 5, 1, None) == C["FVF_OK"]            # empty grid
    assert f(None, 4096, 8, 8, 0.1, 1, 1, None) == C["FVF_ERR_NULL"]
    assert f(4100, 8192, 8, 8, 0.1, 1, 1, None) == C["FVF_ERR_ALIGN"]     # 4100 % 8 != 0
    # fake addresses: the device-memory check runs before the overlap check
    assert f(4096, 4096 + 8, 8, 8, 0.1, 1, 1, None) == C["FVF_ERR_NOT_DEVICE"]


def test_host_memory_rejected(lib):
    """A host (numpy) buffer is not device memory: rejected before launch."""
    u = np.zeros(64, dtype=np.float64)
    v = np.zeros(64, dtype=np.float64)
    st = lib.diffuse2d_step(u.ctypes.data, v.ctypes.data, 8, 8, 0.1, 1, 1, None)
    assert st == C["FVF_ERR_NOT_DEVICE"]


def test_pack_validation(lib):
    f = lib.weno_pack
    vp = ctypes.c_void_p
    table = (vp * 2)(4096, 8192)
    ext = E3(3, 4, 5)
    assert f(table, 2, None, 1, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f(table, 2, ext, 1, 3, 65536, None) == C["FVF_ERR_DIR"]
    assert f(table, 2, ext, 1, -1, 65536, None) == C["FVF_ERR_DIR"]
    assert f(table, 65, ext, 1, 0, 65536, None) == C["FVF_ERR_NV"]
    assert f(table, -1, ext, 1, 0, 65536, None) == C["FVF_ERR_NV"]
    assert f(table, 2, ext, -1, 0, 65536, None) == C["FVF_ERR_SIZE"]
    assert f(table, 2, E3(3, -4, 5), 1, 0, 65536, None) == C["FVF_ERR_SIZE"]
    assert f(table, 0, ext, 1, 0, None, None) == C["FVF_OK"]
    assert f(table, 2, E3(3, 0, 5), 1, 0, None, None) == C["FVF_OK"]
    assert f(table, 2, ext, 1, 0, None, None) == C["FVF_ERR_NULL"]
    assert f(None, 2, ext, 1, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f((vp * 2)(4096, None), 2, ext, 1, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f(table, 2, ext, 1, 0, 65540, None) == C["FVF_ERR_ALIGN"]
    assert f((vp * 2)(4100, 8192), 2, ext, 1, 0, 65536, None) == C["FVF_ERR_ALIGN"]
    assert f(table, 2, ext, 1, 0, 4096 + 800, None) == C["FVF_ERR_NOT_DEVICE"]


def test_rhs_validation(lib):
    f = lib.advect_rhs
    ext = E3(3, 4, 5)
    assert f(4096, 8192, 2, None, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f(4096, 8192, 2, ext, 3, 65536, None) == C["FVF_ERR_DIR"]
    assert f(4096, 8192, 65, ext, 0, 65536, None) == C["FVF_ERR_NV"]
    assert f(4096, 8192, 2, E3(-3, 4, 5), 0, 65536, None) == C["FVF_ERR_SIZE"]
    assert f(4096, 8192, 0, ext, 0, None, None) == C["FVF_OK"]
    assert f(None, 8192, 2, ext, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f(4096, None, 2, ext, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert f(4096, 8192, 2, ext, 0, None, None) == C["FVF_ERR_NULL"]
    assert f(4097, 8192, 2, ext, 0, 65536, None) == C["FVF_ERR_ALIGN"]
    assert f(4096, 65536, 2, ext, 0, 4096 + 640, None) == C["FVF_ERR_NOT_DEVICE"]


def test_unpack_and_rhs_add_validation(lib):
    u, a = lib.flux_unpack, lib.advect_rhs_add
    ext = E3(3, 4, 5)
    assert u(4096, 2, None, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert u(4096, 2, ext, 3, 65536, None) == C["FVF_ERR_DIR"]
    assert u(4096, 65, ext, 0, 65536, None) == C["FVF_ERR_NV"]
    assert u(4096, 2, E3(3, -1, 5), 0, 65536, None) == C["FVF_ERR_SIZE"]
    assert u(None, 0, ext, 0, None, None) == C["FVF_OK"]
    assert u(None, 2, E3(3, 0, 5), 1, None, None) == C["FVF_OK"]
    assert u(None, 2, ext, 0, 65536, None) == C["FVF_ERR_NULL"]
    assert u(4100, 2, ext, 0, 65536, None) == C["FVF_ERR_ALIGN"]
    assert u(4096, 2, ext, 0, 65536, None) == C["FVF_ERR_NOT_DEVICE"]
    assert a(4096, 8192, 2, ext, 3, 65536, None) == C["FVF_ERR_DIR"]
    assert a(4096, 8192, 0, ext, 0, None, None) == C["FVF_OK"]
    assert a(4096, 8192, 2, ext, 0, None, None) == C["FVF_ERR_NULL"]
    assert a(4096, 8192, 2, ext, 0, 65536, None) == C["FVF_ERR_NOT_DEVICE"]


def test_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    u = torch.zeros(8, 8, dtype=torch.float64)
    with pytest.raises(ValueError):
        api.diffuse2d_step(u, u.clone(), 8, 8, 0.1, 1, stream=0)


def test_launch_count_starts_at_zero_without_launches(lib):
    assert api.launch_count() >= 0


def test_copy_validation(lib):
    c, pc = lib.fields_copy, lib.weno_pack_copy
    vp = ctypes.c_void_p
    src = (vp * 2)(4096, 8192)
    dst = (vp * 2)(16384, 32768)
    ext = E3(3, 4, 5)
    assert c(src, 2, None, 1, dst, None) == C["FVF_ERR_NULL"]
    assert c(src, 65, ext, 1, dst, None) == C["FVF_ERR_NV"]
    assert c(src, 2, ext, -1, dst, None) == C["FVF_ERR_SIZE"]
    assert c(src, 2, E3(3, -4, 5), 1, dst, None) == C["FVF_ERR_SIZE"]
    assert c(None, 0, ext, 1, None, None) == C["FVF_OK"]
    assert c(None, 2, E3(3, 0, 5), 1, None, None) == C["FVF_OK"]
    assert c(None, 2, ext, 1, dst, None) == C["FVF_ERR_NULL"]
    assert c(src, 2, ext, 1, None, None) == C["FVF_ERR_NULL"]
    assert c(src, 2, ext, 1, (vp * 2)(16384, None), None) == C["FVF_ERR_NULL"]
    assert c(src, 2, ext, 1, (vp * 2)(16384, 32772), None) == C["FVF_ERR_ALIGN"]
    assert c((vp * 2)(4100, 8192), 2, ext, 1, dst, None) == C["FVF_ERR_ALIGN"]
    assert c(src, 2, ext, 1, dst, None) == C["FVF_ERR_NOT_DEVICE"]
    assert pc(src, 2, None, 1, 0, 65536, dst, None) == C["FVF_ERR_NULL"]
    assert pc(src, 2, ext, 1, 3, 65536, dst, None) == C["FVF_ERR_DIR"]
    assert pc(src, 65, ext, 1, 0, 65536, dst, None) == C["FVF_ERR_NV"]
    assert pc(src, 2, ext, -2, 0, 65536, dst, None) == C["FVF_ERR_SIZE"]
    assert pc(None, 0, ext, 1, 0, None, None, None) == C["FVF_OK"]
    assert pc(src, 2, ext, 1, 0, None, dst, None) == C["FVF_ERR_NULL"]
    assert pc(src, 2, ext, 1, 0, 65536, None, None) == C["FVF_ERR_NULL"]
    assert pc(src, 2, ext, 1, 0, 65540, dst, None) == C["FVF_ERR_ALIGN"]
    assert pc(src, 2, ext, 1, 1, 65536, (vp * 2)(16385, 32768), None) == C["FVF_ERR_ALIGN"]
    assert pc(src, 2, ext, 1, 2, 65536, dst, None) == C["FVF_ERR_NOT_DEVICE"]


def test_stage_validation(lib):
    ax, st = lib.ssprk3_axpby, lib.ssprk3_stage
    vp = ctypes.c_void_p
    ext = E3(3, 4, 5)
    fl = (vp * 3)(4096, 8192, None)
    w = (vp * 3)(16384, 16448, None)
    assert ax(4096, 4096, 8192, 2, None, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NULL"]
    assert ax(4096, 4096, 8192, 65, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NV"]
    assert ax(4096, 4096, 8192, 2, E3(3, -4, 5), 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_SIZE"]
    assert ax(4096, 4096, 8192, 2, ext, float("nan"), 0.25, 0.1, 65536, None) == C["FVF_ERR_ALPHA"]
    assert ax(4096, 4096, 8192, 2, ext, 0.75, float("inf"), 0.1, 65536, None) == C["FVF_ERR_ALPHA"]
    assert ax(4096, 4096, 8192, 2, ext, 0.75, 0.25, float("-inf"), 65536, None) == C["FVF_ERR_ALPHA"]
    assert ax(None, None, None, 0, ext, 0.75, 0.25, 0.1, None, None) == C["FVF_OK"]
    assert ax(None, None, None, 2, E3(3, 0, 5), 0.75, 0.25, 0.1, None, None) == C["FVF_OK"]
    assert ax(None, 4096, 8192, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NULL"]
    assert ax(4096, 4096, None, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NULL"]
    assert ax(4096, 4096, 8192, 2, ext, 0.75, 0.25, 0.1, None, None) == C["FVF_ERR_NULL"]
    assert ax(4096, 4100, 8192, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_ALIGN"]
    assert ax(4096, 4096, 8192, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NOT_DEVICE"]
    assert st(4096, 4096, fl, w, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NOT_DEVICE"]
    assert st(4096, 4096, None, w, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NULL"]
    assert st(4096, 4096, fl, None, 2, ext, 0.75, 0.25, 0.1, 65536, None) == C["FVF_ERR_NULL"]
    assert st(4096, 4096, (vp * 3)(None, 8192, None), w, 2, ext, 0.75, 0.25, 0.1, 65536,
              None) == C["FVF_ERR_NULL"]
    assert st(4096, 4096, (vp * 3)(4096, 8192, 12288), w, 2, ext, 0.75, 0.25, 0.1, 65536,
              None) == C["FVF_ERR_NULL"]   # z flux given without its inverse widths
    assert st(4096, 4096, fl, (vp * 3)(16384, 16452, None), 2, ext, 0.75, 0.25, 0.1, 65536,
              None) == C["FVF_ERR_ALIGN"]
    assert st(4096, 4096, fl, w, 2, ext, 0.75, 0.25, float("nan"), 65536, None) == \
        C["FVF_ERR_ALPHA"]


def test_diffuse3d_validation(lib):
    f = lib.diffuse3d_step
    assert f(4096, 8192, 4, 4, 4, 0.1, 1, 2, None) == C["FVF_ERR_DTYPE"]
    assert f(4096, 8192, 4, -4, 4, 0.1, 1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(4096, 8192, 4, 4, 4, 0.1, -1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(4096, 8192, 1 << 40, 1 << 40, 4, 0.1, 1, 1, None) == C["FVF_ERR_SIZE"]
    assert f(4096, 8192, 4, 4, 4, float("nan"), 1, 1, None) == C["FVF_ERR_ALPHA"]
    assert f(4096, 8192, 4, 4, 4, 1e300, 1, 0, None) == C["FVF_ERR_ALPHA"]
    assert f(None, None, 4, 0, 4, 0.1, 1, 1, None) == C["FVF_OK"]
    assert f(None, None, 4, 4, 4, 0.1, 0, 1, None) == C["FVF_OK"]
    assert f(None, 8192, 4, 4, 4, 0.1, 1, 1, None) == C["FVF_ERR_NULL"]
    assert f(4100, 8192, 4, 4, 4, 0.1, 1, 1, None) == C["FVF_ERR_ALIGN"]
    assert f(4096, 8192, 4, 4, 4, 0.1, 1, 1, None) == C["FVF_ERR_NOT_DEVICE"]


def test_device_error_flag_call(lib):
    """NULL is refused; without a usable GPU the read reports a CUDA error,
    with one it reads 0 (no kernel has set the flag)."""
    assert lib.fvf_device_error(None) == C["FVF_ERR_NULL"]
    flag = ctypes.c_int(7)
    st = lib.fvf_device_error(ctypes.byref(flag))
    assert (st, flag.value) in ((C["FVF_ERR_CUDA"], 0), (C["FVF_OK"], 0))


def test_fp32_pack_and_flux_validation(lib):
    vp = ctypes.c_void_p
    ext = E3(3, 4, 5)
    p, a, aa = lib.weno_pack_f32, lib.advect_rhs_f32, lib.advect_rhs_add_f32
    table = (vp * 2)(4096, 8192)
    assert p(table, 2, ext, 1, 3, 65536, None) == C["FVF_ERR_DIR"]
    assert p(table, 2, ext, 1, 0, 65538, None) == C["FVF_ERR_ALIGN"]
    assert p((vp * 2)(4098, 8192), 2, ext, 1, 0, 65536, None) == C["FVF_ERR_ALIGN"]
    assert p(table, 2, ext, 1, 0, 65540, None) == C["FVF_ERR_NOT_DEVICE"]   # 4-byte aligned
    for f in (a, aa):
        assert f(4096, 8192, 2, ext, 3, 65536, None) == C["FVF_ERR_DIR"]
        assert f(4096, 8192, 0, ext, 0, None, None) == C["FVF_OK"]
        assert f(4098, 8192, 2, ext, 0, 65536, None) == C["FVF_ERR_ALIGN"]
        assert f(4100, 8196, 2, ext, 0, 65540, None) == C["FVF_ERR_NOT_DEVICE"]


def test_degenerate_sizes_are_valid_calls(lib):
    """The boundary accepts, as valid calls, sizes a narrower contract could
    reject: empty grids, nv = 0 and zero extents return FVF_OK without
    touching memory (NULL pointers are fine then, and nothing is launched);
    grids with no interior (nx or ny <= 2) and a swept axis of extent 1 are
    ordinary calls, which proceed to the pointer checks (FVF_ERR_NULL here,
    not FVF_ERR_SIZE).  Their results are pinned on the GPU
    (test_gpu_degenerate.py)."""
    before = lib.fvf_launch_count()
    d2, d3 = lib.diffuse2d_step, lib.diffuse3d_step
    for dt in (0, 1):
        assert d2(None, None, 0, 9, 0.1, 3, dt, None) == C["FVF_OK"]
        assert d2(None, None, 9, 0, 0.1, 3, dt, None) == C["FVF_OK"]
        assert d3(None, None, 9, 0, 9, 0.1, 3, dt, None) == C["FVF_OK"]
        for nx, ny in ((1, 1), (2, 2), (2, 9), (9, 1)):
            assert d2(None, None, nx, ny, 0.1, 1, dt, None) == C["FVF_ERR_NULL"]
    ext0 = E3(0, 5, 5)
    ext1 = E3(5, 5, 1)
    tab = (ctypes.c_void_p * 1)(None)
    assert lib.weno_pack(tab, 0, E3(5, 5, 5), 2, 0, None, None) == C["FVF_OK"]
    assert lib.weno_pack(tab, 1, ext0, 2, 0, None, None) == C["FVF_OK"]
    assert lib.weno_pack(tab, 1, ext1, 2, 2, None, None) == C["FVF_ERR_NULL"]
    for name in ("advect_rhs", "advect_rhs_add"):
        f = getattr(lib, name)
        assert f(None, None, 0, E3(5, 5, 5), 0, None, None) == C["FVF_OK"]
        assert f(None, None, 2, ext0, 1, None, None) == C["FVF_OK"]
        assert f(None, None, 2, ext1, 2, None, None) == C["FVF_ERR_NULL"]
    assert lib.flux_unpack(None, 0, E3(5, 5, 5), 1, None, None) == C["FVF_OK"]
    assert lib.fields_copy(tab, 0, E3(5, 5, 5), 1, tab, None) == C["FVF_OK"]
    assert lib.fvf_launch_count() == before
