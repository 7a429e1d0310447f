"""The benchmark's ablation kernels (one thread per cell-variable pair, the
mapping MFC pull request #2087 replaces) compute the same x pack and x flux
difference as the oracle, bit for bit, so the timing comparison in bench.py
compares equal work."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import inputs
from tests.gpu_util import assert_bits_equal, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def _lib():
    import bench
    return bench.load_ablation()


@pytest.mark.parametrize("extents,g,nv", [((5, 4, 3), 2, 3), ((33, 31, 7), 3, 8),
                                          ((40, 1, 1), 1, 2), ((6, 9, 1), 2, 7)])
def test_collapse4_pack_and_rhs_match_oracle(extents, g, nv):
    torch = torch_cuda()
    lib = _lib()
    ext = (ctypes.c_int64 * 3)(*extents)
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    dev = [to_dev(f) for f in fields]
    M = oracle.pack_extents(extents, g, 0)
    out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float64, device="cuda")
    table = (ctypes.c_void_p * nv)(*[d.data_ptr() for d in dev])
    assert lib.ablation_pack_x_collapse4(table, nv, ext, g, out.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert_bits_equal(to_host(out), oracle.weno_pack(fields, extents, g, 0))
    flux = inputs.face_fluxes(inputs.config_seed(4), nv, extents, 0)
    w = inputs.inverse_spacing(inputs.config_seed(4), extents[0])
    rhs = torch.empty(int(np.prod(extents)) * nv, dtype=torch.float64, device="cuda")
    assert lib.ablation_rhs_x_collapse4(None, None, nv, ext, None, None) == 1
    df, dw = to_dev(flux), to_dev(w)
    assert lib.ablation_rhs_x_collapse4(df.data_ptr(), dw.data_ptr(), nv, ext, rhs.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert_bits_equal(to_host(rhs), oracle.advect_rhs(flux, w, nv, extents, 0))
