"""Helpers for the GPU parity tests: device transfers and exact comparisons."""
from __future__ import annotations

import numpy as np


def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("these tests need a CUDA GPU")
    from finite_volume_field_gb300 import buildlib
    buildlib.build()
    return torch


def to_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_bits_equal(got: np.ndarray, want: np.ndarray, nan_payloads: bool = True, what=""):
    """Bit-for-bit equality.  With ``nan_payloads`` False, NaNs match NaNs
    whatever their payload (arithmetic does not preserve payloads)."""
    got = np.ascontiguousarray(got).reshape(-1)
    want = np.ascontiguousarray(want).reshape(-1)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    ui = np.uint64 if got.dtype == np.float64 else np.uint32
    gb, wb = got.view(ui), want.view(ui)
    diff = gb != wb
    if not nan_payloads:
        diff &= ~(np.isnan(got) & np.isnan(want))
    if diff.any():
        idx = np.flatnonzero(diff)
        k = idx[0]
        raise AssertionError(
            f"{what}: {idx.size} of {got.size} elements differ; first at {k}: "
            f"got {got[k]!r} ({int(gb[k]):#x}) want {want[k]!r} ({int(wb[k]):#x})")


def guarded(torch, n: int, dtype, pad: int = 64):
    """A device tensor of n elements followed by ``pad`` canary elements
    (a NaN bit pattern).  Returns (whole, view_of_first_n)."""
    whole = torch.empty(n + pad, dtype=dtype, device="cuda")
    if dtype == torch.float64:
        whole.view(torch.int64)[n:] = 0x7FF4A5A5A5A5A5A5
    else:
        whole.view(torch.int32)[n:] = 0x7FA5A5A5
    return whole, whole[:n]


def canary_intact(torch, whole, n: int) -> bool:
    tail = whole[n:]
    if whole.dtype == torch.float64:
        return bool((tail.view(torch.int64) == 0x7FF4A5A5A5A5A5A5).all())
    return bool((tail.view(torch.int32) == 0x7FA5A5A5).all())
