"""GB300-native per-cell field sweeps: 2D 5-point and 3D 7-point diffusion
with ping-pong buffers, the multi-variable WENO input pack and the finite-volume
flux-difference source (assigned or accumulated), the directional flux
copy back to the physical frame, the conservative-variable copy (alone or
fused with the pack) and the SSPRK3 stage update (alone or fused with the
flux difference), as sm_103a CUDA kernels behind a C ABI
(include/fvf.h, libfvf.so).

The public calls are re-exported from ``api``; they load libfvf.so on first
use and raise if it is missing.  ``inputs`` holds the seeded synthetic input
generators.
"""
from .api import (FVF_FP32, FVF_FP64, MAX_NV, FvfError, advect_rhs, advect_rhs_add,
                  advect_rhs_add_f32, advect_rhs_f32, device_error, diffuse2d_step,
                  diffuse3d_step, fields_copy, flux_unpack, last_cuda_error, launch_count, load,
                  ssprk3_axpby, ssprk3_stage, status_string, weno_pack, weno_pack_copy,
                  weno_pack_f32)

__all__ = ["FVF_FP32", "FVF_FP64", "MAX_NV", "FvfError", "advect_rhs", "advect_rhs_add",
           "advect_rhs_add_f32", "advect_rhs_f32", "device_error", "diffuse2d_step",
           "diffuse3d_step", "fields_copy", "flux_unpack", "last_cuda_error", "launch_count",
           "load", "ssprk3_axpby", "ssprk3_stage", "status_string", "weno_pack",
           "weno_pack_copy", "weno_pack_f32"]
