// fvf_internal.cuh -- launchers shared between the C-ABI layer (fvf_abi.cu)
// and the kernel files.  Not part of the public interface (include/fvf.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Index checks for debug builds.  Built with -DFVF_BOUNDS_CHECK=1 (for
// small grids; buildlib.build(bounds_check=True) makes libfvf_check.so),
// FVF_IN(i, n) tests a global index against the extent of the array it
// addresses before the access it guards; a failing test records itself in
// the translation unit's flag (read through fvf_device_error) and the access
// is skipped -- nothing traps.  In release builds FVF_IN is the constant true
// and the generated code is unchanged.
#ifndef FVF_BOUNDS_CHECK
#define FVF_BOUNDS_CHECK 0
#endif
#if FVF_BOUNDS_CHECK
static __device__ int g_bounds_failed;
static __device__ __forceinline__ bool fvf_in_bounds(int64_t i, int64_t n) {
    if (i >= 0 && i < n) return true;
    atomicExch(&g_bounds_failed, 1);
    return false;
}
#define FVF_IN(i, n) fvf_in_bounds((int64_t)(i), (int64_t)(n))
#define FVF_BOUNDS_READER(fn)                                                    \
    cudaError_t fn(int *failed) {                                                \
        int zero = 0;                                                            \
        cudaError_t e = cudaMemcpyFromSymbol(failed, g_bounds_failed, sizeof(int)); \
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bounds_failed, &zero, sizeof(int)); \
        return e;                                                                \
    }
#else
#define FVF_IN(i, n) true
#define FVF_BOUNDS_READER(fn)     \
    cudaError_t fn(int *failed) { \
        *failed = 0;              \
        return cudaSuccess;       \
    }
#endif

namespace fvf {

constexpr int kMaxNv = 64;

// Pointer table of the pack's input fields (FP64 or FP32 elements, as the
// launch says), passed to the kernel by value (kernel parameter space), so
// concurrent calls never share state.
struct FieldTable {
    const void *p[kMaxNv];
};

// Output pointer table of the conservative-variable copies (one array per
// variable, each the size of the stored box), passed by value like FieldTable.
struct CopyTable {
    double *p[kMaxNv];
};

// Box geometry of a 3D sweep: interior extents n, stored extents N (n + 2g on
// axes with n > 1, else 1) and ghost offsets g (g where n > 1, else 0).
struct Box {
    int64_t n[3];
    int64_t N[3];
    int64_t g[3];
};

// Arguments of the SSPRK3 stage update, alone (f[0] = rhs) or fused with the
// flux difference (f[0..2] = x/y/z face fluxes, y and z possibly NULL;
// w[0..2] = inverse spacings of the present directions).  Cell arrays have
// n[0]*n[1]*n[2] cells per variable, j fastest, the variable slowest.
struct RkStageArgs {
    const double *u0;
    const double *u;
    const double *f[3];
    const double *w[3];
    double *out;
    int nv;
    int64_t n[3];
    double a, b, dt;
};

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Index of the current device in the per-device caches of the launchers
// (0..63; devices beyond 63 share the last slot).
int device_slot();

// Each launcher enqueues its kernels on `stream`, adds the number of kernels
// it launched to *launches and returns the first launch error (cudaSuccess
// if none).  Arguments have already been validated by the caller.
cudaError_t launch_diffuse2d(void *u, void *v, int64_t nx, int64_t ny, double alpha,
                             int64_t nsteps, bool fp64, cudaStream_t stream,
                             uint64_t *launches);

cudaError_t launch_diffuse3d(void *u, void *v, int64_t nx, int64_t ny, int64_t nz, double alpha,
                             int64_t nsteps, bool fp64, cudaStream_t stream,
                             uint64_t *launches);

// Reads and clears the device flag that kernels with bounded waits set when
// a wait expires (synchronises the device).
cudaError_t read_device_error(int *flag);

// Each kernel file's index-check flag (always 0 unless built with
// FVF_BOUNDS_CHECK); reading clears it.
cudaError_t read_bounds_diffuse2d(int *failed);
cudaError_t read_bounds_diffuse3d(int *failed);
cudaError_t read_bounds_pack(int *failed);
cudaError_t read_bounds_rhs(int *failed);
cudaError_t read_bounds_rk(int *failed);

cudaError_t launch_weno_pack(const FieldTable &fields, int nv, const Box &box, int dir,
                             void *out, bool fp32, cudaStream_t stream, uint64_t *launches);

// The conservative-variable copy alone: copy_i[e] = field_i[e] for the
// `stored` elements of every variable.
cudaError_t launch_fields_copy(const FieldTable &fields, int nv, int64_t stored,
                               const CopyTable &copies, cudaStream_t stream, uint64_t *launches);

// The pack fused with the conservative-variable copy: one pass reads every
// stored element once, writes it to its copy and, inside the pack region, to
// the packed output.
cudaError_t launch_weno_pack_copy(const FieldTable &fields, int nv, const Box &box, int dir,
                                  double *out, const CopyTable &copies, cudaStream_t stream,
                                  uint64_t *launches);

cudaError_t launch_rk_stage(const RkStageArgs &args, bool fused, cudaStream_t stream,
                            uint64_t *launches);

cudaError_t launch_advect_rhs(const void *flux, const void *inv_d, int nv, const int64_t n[3],
                              int dir, bool accumulate, bool fp32, void *rhs,
                              cudaStream_t stream, uint64_t *launches);

}  // namespace fvf
