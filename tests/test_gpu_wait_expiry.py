"""The bounded mbarrier wait gives up on a phase that cannot complete.

Kernels that wait on their own asynchronous copies (the FP32 3D diffusion
kernel) bound every wait.  This test builds a one-kernel program on the
shared helper header: a barrier that expects two arrivals gets one, the wait
must return false after its poll limit (no fault, no hang), and after the
second arrival the same wait must succeed.  The context stays usable."""
from __future__ import annotations

import ctypes
import subprocess
from pathlib import Path

import pytest

from tests.gpu_util import torch_cuda

pytestmark = pytest.mark.gpu

HERE = Path(__file__).resolve().parent


def test_bounded_wait_expires_and_recovers(tmp_path):
    torch = torch_cuda()
    from finite_volume_field_gb300 import buildlib
    so = tmp_path / "libwaitcheck.so"
    subprocess.run([buildlib.nvcc(), "-O2", "-std=c++17", *buildlib.ARCH, "-Xcompiler", "-fPIC",
                    "-shared", "-cudart", "static", str(HERE / "wait_expiry_check.cu"), "-o",
                    str(so)], check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    lib.run_wait_expiry.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_uint]
    status = (ctypes.c_int * 2)(0, 0)
    assert lib.run_wait_expiry(status, 4096) == 0
    assert list(status) == [2, 1]
    # the device still runs work afterwards
    x = torch.arange(1000, dtype=torch.float64, device="cuda")
    assert float(x.sum()) == 499500.0
