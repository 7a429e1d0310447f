// fvf_abi.cu -- the extern "C" entry points declared in include/fvf.h:
// argument validation on the host, then dispatch to the kernel launchers.
//
// Nothing is launched unless every argument passed validation.  Beyond the
// arithmetic checks (sizes, alignment, overlap), every array pointer is
// checked to be device memory of the current device and, through the driver's
// cuMemGetAddressRange, to lie with its whole extent inside one allocation, so
// a wrong size or a host pointer becomes a status code instead of a device
// fault.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fvf.h"
#include "fvf_internal.cuh"

#define FVF_API extern "C" __attribute__((visibility("default")))

namespace fvf {

static std::atomic<uint64_t> g_launches{0};
static thread_local int g_last_cuda_error = 0;

int device_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return 0;
    }
    return dev < 63 ? dev : 63;
}

int sm_count() {
    static std::atomic<int> cached[64];   // concurrent first calls store the same value
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 152;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

namespace {

using GetRangeFn = CUresult (*)(CUdeviceptr *, size_t *, CUdeviceptr);

GetRangeFn get_range_fn() {
    static std::once_flag once;
    static GetRangeFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetRangeFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Checks that [p, p + bytes) is device (or managed) memory of the current
// device inside a single allocation.
int check_device_array(const void *p, uint64_t bytes) {
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof(a));
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return FVF_ERR_NOT_DEVICE;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return FVF_ERR_NOT_DEVICE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || a.device != dev) return FVF_ERR_NOT_DEVICE;
    if (GetRangeFn fn = get_range_fn()) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (fn(&base, &size, (CUdeviceptr)(uintptr_t)p) != CUDA_SUCCESS) return FVF_ERR_NOT_DEVICE;
        const uint64_t off = (uint64_t)((uintptr_t)p - (uintptr_t)base);
        if (off > size || bytes > size - off) return FVF_ERR_RANGE;
    }
    return FVF_OK;
}

bool overlaps(const void *a, uint64_t abytes, const void *b, uint64_t bbytes) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// a*b with overflow check against a cap (products of sizes, in elements).
bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    const int64_t cap = (int64_t)1 << 60;
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > cap / a) return false;
    *out = a * b;
    return true;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FVF_OK;
    g_last_cuda_error = (int)e;
    return FVF_ERR_CUDA;
}

}  // namespace
}  // namespace fvf

using namespace fvf;

FVF_API int diffuse2d_step(void *u, void *v, int64_t nx, int64_t ny, double alpha,
                           int64_t nsteps, int dtype, void *stream) {
    if (dtype != FVF_FP32 && dtype != FVF_FP64) return FVF_ERR_DTYPE;
    if (nx < 0 || ny < 0 || nsteps < 0) return FVF_ERR_SIZE;
    int64_t cells = 0;
    if (!mul_ok(nx, ny, &cells)) return FVF_ERR_SIZE;
    if (!std::isfinite(alpha)) return FVF_ERR_ALPHA;
    if (dtype == FVF_FP32 && !std::isfinite((float)alpha)) return FVF_ERR_ALPHA;
    if (cells == 0 || nsteps == 0) return FVF_OK;
    if (!u || !v) return FVF_ERR_NULL;
    const uint64_t esize = dtype == FVF_FP64 ? 8 : 4;
    if ((uintptr_t)u % esize || (uintptr_t)v % esize) return FVF_ERR_ALIGN;
    const uint64_t bytes = (uint64_t)cells * esize;
    int st = check_device_array(u, bytes);
    if (st == FVF_OK) st = check_device_array(v, bytes);
    if (st != FVF_OK) return st;
    if (overlaps(u, bytes, v, bytes)) return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e = launch_diffuse2d(u, v, nx, ny, alpha, nsteps, dtype == FVF_FP64,
                                           (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API int diffuse3d_step(void *u, void *v, int64_t nx, int64_t ny, int64_t nz, double alpha,
                           int64_t nsteps, int dtype, void *stream) {
    if (dtype != FVF_FP32 && dtype != FVF_FP64) return FVF_ERR_DTYPE;
    if (nx < 0 || ny < 0 || nz < 0 || nsteps < 0) return FVF_ERR_SIZE;
    int64_t t = 0, cells = 0;
    if (!mul_ok(nx, ny, &t) || !mul_ok(t, nz, &cells)) return FVF_ERR_SIZE;
    if (!std::isfinite(alpha)) return FVF_ERR_ALPHA;
    if (dtype == FVF_FP32 && !std::isfinite((float)alpha)) return FVF_ERR_ALPHA;
    if (cells == 0 || nsteps == 0) return FVF_OK;
    if (!u || !v) return FVF_ERR_NULL;
    const uint64_t esize = dtype == FVF_FP64 ? 8 : 4;
    if ((uintptr_t)u % esize || (uintptr_t)v % esize) return FVF_ERR_ALIGN;
    const uint64_t bytes = (uint64_t)cells * esize;
    int st = check_device_array(u, bytes);
    if (st == FVF_OK) st = check_device_array(v, bytes);
    if (st != FVF_OK) return st;
    if (overlaps(u, bytes, v, bytes)) return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e = launch_diffuse3d(u, v, nx, ny, nz, alpha, nsteps, dtype == FVF_FP64,
                                           (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

// Shared validation and launch of weno_pack (FP64) and weno_pack_f32.
static int weno_pack_impl(const void *const *fields, int nv, const int64_t extents[3], int ghost,
                          int dir, void *out, bool fp32, void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (dir < 0 || dir > 2) return FVF_ERR_DIR;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    if (ghost < 0) return FVF_ERR_SIZE;
    Box box;
    for (int a = 0; a < 3; ++a) {
        if (extents[a] < 0) return FVF_ERR_SIZE;
        box.n[a] = extents[a];
        box.g[a] = extents[a] > 1 ? ghost : 0;
        box.N[a] = extents[a] > 1 ? extents[a] + 2 * (int64_t)ghost : extents[a];
    }
    int64_t stored = 0, t = 0, cells_out = 0, elems_out = 0;
    if (!mul_ok(box.N[0], box.N[1], &t) || !mul_ok(t, box.N[2], &stored)) return FVF_ERR_SIZE;
    const int64_t M[3][3] = {{box.N[0], box.n[1], box.n[2]},
                             {box.N[1], box.n[0], box.n[2]},
                             {box.N[2], box.n[1], box.n[0]}};
    if (!mul_ok(M[dir][0], M[dir][1], &t) || !mul_ok(t, M[dir][2], &cells_out) ||
        !mul_ok(cells_out, nv, &elems_out))
        return FVF_ERR_SIZE;
    if (elems_out == 0) return FVF_OK;
    if (!fields || !out) return FVF_ERR_NULL;
    const uint64_t esize = fp32 ? 4 : 8;
    if ((uintptr_t)out % esize) return FVF_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)elems_out * esize, in_bytes = (uint64_t)stored * esize;
    FieldTable table;
    std::memset(&table, 0, sizeof(table));
    for (int i = 0; i < nv; ++i) {
        if (!fields[i]) return FVF_ERR_NULL;
        if ((uintptr_t)fields[i] % esize) return FVF_ERR_ALIGN;
        table.p[i] = fields[i];
    }
    int st = check_device_array(out, out_bytes);
    for (int i = 0; i < nv && st == FVF_OK; ++i) st = check_device_array(fields[i], in_bytes);
    if (st != FVF_OK) return st;
    for (int i = 0; i < nv; ++i)
        if (overlaps(fields[i], in_bytes, out, out_bytes)) return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e =
        launch_weno_pack(table, nv, box, dir, out, fp32, (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API int weno_pack(const double *const *fields, int nv, const int64_t extents[3], int ghost,
                      int dir, double *out, void *stream) {
    return weno_pack_impl(reinterpret_cast<const void *const *>(fields), nv, extents, ghost, dir,
                          out, false, stream);
}

FVF_API int weno_pack_f32(const float *const *fields, int nv, const int64_t extents[3],
                          int ghost, int dir, float *out, void *stream) {
    return weno_pack_impl(reinterpret_cast<const void *const *>(fields), nv, extents, ghost, dir,
                          out, true, stream);
}

// Pointer tables of the multi-variable calls: each entry non-NULL and 8-byte
// aligned; fills *table (a FieldTable or CopyTable).
template <typename Table, typename Ptr>
static int fill_table(Ptr const *ptrs, int nv, Table *table) {
    if (!ptrs) return FVF_ERR_NULL;
    std::memset(table, 0, sizeof(*table));
    for (int i = 0; i < nv; ++i) {
        if (!ptrs[i]) return FVF_ERR_NULL;
        if ((uintptr_t)ptrs[i] % 8) return FVF_ERR_ALIGN;
        table->p[i] = ptrs[i];
    }
    return FVF_OK;
}

// Every entry of a table is `bytes` of device memory of this device.
template <typename Ptr>
static int check_device_table(Ptr const *ptrs, int nv, uint64_t bytes) {
    for (int i = 0; i < nv; ++i) {
        const int st = check_device_array(ptrs[i], bytes);
        if (st != FVF_OK) return st;
    }
    return FVF_OK;
}

// A copy must overlap no field, no other copy and not out (out_bytes == 0:
// no out).
static bool copies_overlap(const double *const *fields, double *const *copies, int nv,
                           uint64_t bytes, const double *out, uint64_t out_bytes) {
    for (int i = 0; i < nv; ++i) {
        for (int k = 0; k < nv; ++k) {
            if (overlaps(copies[i], bytes, fields[k], bytes)) return true;
            if (k != i && overlaps(copies[i], bytes, copies[k], bytes)) return true;
        }
        if (out_bytes && overlaps(copies[i], bytes, out, out_bytes)) return true;
    }
    return false;
}

// Stored box of interior extents with ghost width `ghost`; *stored gets
// N1*N2*N3.  FVF_OK or the status of the first bad argument.
static int make_box(const int64_t extents[3], int ghost, Box *box, int64_t *stored) {
    if (!extents) return FVF_ERR_NULL;
    if (ghost < 0) return FVF_ERR_SIZE;
    for (int a = 0; a < 3; ++a) {
        if (extents[a] < 0) return FVF_ERR_SIZE;
        box->n[a] = extents[a];
        box->g[a] = extents[a] > 1 ? ghost : 0;
        box->N[a] = extents[a] > 1 ? extents[a] + 2 * (int64_t)ghost : extents[a];
    }
    int64_t t = 0;
    if (!mul_ok(box->N[0], box->N[1], &t) || !mul_ok(t, box->N[2], stored)) return FVF_ERR_SIZE;
    return FVF_OK;
}

FVF_API int fields_copy(const double *const *fields, int nv, const int64_t extents[3], int ghost,
                        double *const *copies, void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    Box box;
    int64_t stored = 0, elems = 0;
    int st = make_box(extents, ghost, &box, &stored);
    if (st != FVF_OK) return st;
    if (!mul_ok(stored, nv, &elems)) return FVF_ERR_SIZE;
    if (elems == 0) return FVF_OK;
    const uint64_t bytes = (uint64_t)stored * 8;
    FieldTable ft;
    CopyTable ct;
    st = fill_table(fields, nv, &ft);
    if (st == FVF_OK) st = fill_table(copies, nv, &ct);
    if (st == FVF_OK) st = check_device_table(fields, nv, bytes);
    if (st == FVF_OK) st = check_device_table(copies, nv, bytes);
    if (st != FVF_OK) return st;
    if (copies_overlap(fields, copies, nv, bytes, nullptr, 0)) return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e = launch_fields_copy(ft, nv, stored, ct, (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API int weno_pack_copy(const double *const *fields, int nv, const int64_t extents[3],
                           int ghost, int dir, double *out, double *const *copies,
                           void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (dir < 0 || dir > 2) return FVF_ERR_DIR;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    Box box;
    int64_t stored = 0, t = 0, cells_out = 0, elems_out = 0;
    int st = make_box(extents, ghost, &box, &stored);
    if (st != FVF_OK) return st;
    const int64_t M[3][3] = {{box.N[0], box.n[1], box.n[2]},
                             {box.N[1], box.n[0], box.n[2]},
                             {box.N[2], box.n[1], box.n[0]}};
    if (!mul_ok(M[dir][0], M[dir][1], &t) || !mul_ok(t, M[dir][2], &cells_out) ||
        !mul_ok(cells_out, nv, &elems_out) || !mul_ok(stored, nv, &t))
        return FVF_ERR_SIZE;
    if (elems_out == 0) return FVF_OK;
    if (!out) return FVF_ERR_NULL;
    if ((uintptr_t)out % 8) return FVF_ERR_ALIGN;
    const uint64_t out_bytes = (uint64_t)elems_out * 8, in_bytes = (uint64_t)stored * 8;
    FieldTable ft;
    CopyTable ct;
    st = fill_table(fields, nv, &ft);
    if (st == FVF_OK) st = fill_table(copies, nv, &ct);
    if (st == FVF_OK) st = check_device_array(out, out_bytes);
    if (st == FVF_OK) st = check_device_table(fields, nv, in_bytes);
    if (st == FVF_OK) st = check_device_table(copies, nv, in_bytes);
    if (st != FVF_OK) return st;
    for (int i = 0; i < nv; ++i)
        if (overlaps(fields[i], in_bytes, out, out_bytes)) return FVF_ERR_ALIAS;
    if (copies_overlap(fields, copies, nv, in_bytes, out, out_bytes)) return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e = launch_weno_pack_copy(ft, nv, box, dir, out, ct, (cudaStream_t)stream,
                                                &launched);
    g_launches += launched;
    return cuda_status(e);
}

// out of a stage update may be u or u0 itself (same start; each element is
// read before it is written) but must not overlap them otherwise.
static bool bad_inplace(const double *out, const double *in, uint64_t bytes) {
    return out != in && overlaps(out, bytes, in, bytes);
}

// Shared validation and launch of ssprk3_axpby (rhs given, fused false) and
// ssprk3_stage (fluxes given, fused true).
static int rk_stage_impl(const double *u0, const double *u, const double *rhs,
                         const double *const *flux, const double *const *inv_d, int nv,
                         const int64_t extents[3], double a, double b, double dt, double *out,
                         bool fused, void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    RkStageArgs A;
    std::memset(&A, 0, sizeof(A));
    int64_t t = 0, cells = 0, elems = 0, felems[3] = {0, 0, 0};
    for (int d = 0; d < 3; ++d) {
        if (extents[d] < 0) return FVF_ERR_SIZE;
        A.n[d] = extents[d];
    }
    if (!mul_ok(A.n[0], A.n[1], &t) || !mul_ok(t, A.n[2], &cells) || !mul_ok(cells, nv, &elems))
        return FVF_ERR_SIZE;
    for (int d = 0; d < 3; ++d) {
        int64_t F[3] = {A.n[0], A.n[1], A.n[2]}, faces = 0;
        F[d] += 1;
        if (!mul_ok(F[0], F[1], &t) || !mul_ok(t, F[2], &faces) || !mul_ok(faces, nv, &felems[d]))
            return FVF_ERR_SIZE;
    }
    if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(dt)) return FVF_ERR_ALPHA;
    if (elems == 0) return FVF_OK;
    if (!u0 || !u || !out) return FVF_ERR_NULL;
    if (fused) {
        if (!flux || !inv_d || !flux[0] || !inv_d[0]) return FVF_ERR_NULL;
        for (int d = 0; d < 3; ++d) {
            if (flux[d] && !inv_d[d]) return FVF_ERR_NULL;
            A.f[d] = flux[d];
            A.w[d] = flux[d] ? inv_d[d] : nullptr;
        }
    } else {
        if (!rhs) return FVF_ERR_NULL;
        A.f[0] = rhs;
    }
    const double *ptrs[8] = {u0, u, out, A.f[0], A.f[1], A.f[2], A.w[0], A.w[1]};
    for (const double *p : ptrs)
        if ((uintptr_t)p % 8) return FVF_ERR_ALIGN;
    if ((uintptr_t)A.w[2] % 8) return FVF_ERR_ALIGN;
    const uint64_t cbytes = (uint64_t)elems * 8;
    uint64_t fbytes[3], wbytes[3];
    for (int d = 0; d < 3; ++d) {
        fbytes[d] = fused ? (uint64_t)felems[d] * 8 : (d == 0 ? cbytes : 0);
        wbytes[d] = (uint64_t)A.n[d] * 8;
    }
    int st = check_device_array(u0, cbytes);
    if (st == FVF_OK) st = check_device_array(u, cbytes);
    if (st == FVF_OK) st = check_device_array(out, cbytes);
    for (int d = 0; d < 3 && st == FVF_OK; ++d) {
        if (A.f[d]) st = check_device_array(A.f[d], fbytes[d]);
        if (st == FVF_OK && A.w[d]) st = check_device_array(A.w[d], wbytes[d]);
    }
    if (st != FVF_OK) return st;
    if (bad_inplace(out, u, cbytes) || bad_inplace(out, u0, cbytes)) return FVF_ERR_ALIAS;
    for (int d = 0; d < 3; ++d) {
        if (A.f[d] && overlaps(out, cbytes, A.f[d], fbytes[d])) return FVF_ERR_ALIAS;
        if (A.w[d] && overlaps(out, cbytes, A.w[d], wbytes[d])) return FVF_ERR_ALIAS;
    }
    A.u0 = u0;
    A.u = u;
    A.out = out;
    A.nv = nv;
    A.a = a;
    A.b = b;
    A.dt = dt;
    uint64_t launched = 0;
    const cudaError_t e = launch_rk_stage(A, fused, (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API int ssprk3_axpby(const double *u0, const double *u, const double *rhs, int nv,
                         const int64_t extents[3], double a, double b, double dt, double *out,
                         void *stream) {
    return rk_stage_impl(u0, u, rhs, nullptr, nullptr, nv, extents, a, b, dt, out, false, stream);
}

FVF_API int ssprk3_stage(const double *u0, const double *u, const double *const flux[3],
                         const double *const inv_d[3], int nv, const int64_t extents[3], double a,
                         double b, double dt, double *out, void *stream) {
    return rk_stage_impl(u0, u, nullptr, flux, inv_d, nv, extents, a, b, dt, out, true, stream);
}

static int advect_rhs_impl(const void *flux, const void *inv_d, int nv, const int64_t extents[3],
                           int dir, bool accumulate, bool fp32, void *rhs, void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (dir < 0 || dir > 2) return FVF_ERR_DIR;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    int64_t n[3], F[3];
    for (int a = 0; a < 3; ++a) {
        if (extents[a] < 0) return FVF_ERR_SIZE;
        n[a] = extents[a];
        F[a] = extents[a] + (a == dir ? 1 : 0);
    }
    int64_t t = 0, cells = 0, faces = 0, elems = 0, felems = 0;
    if (!mul_ok(n[0], n[1], &t) || !mul_ok(t, n[2], &cells) || !mul_ok(cells, nv, &elems))
        return FVF_ERR_SIZE;
    if (!mul_ok(F[0], F[1], &t) || !mul_ok(t, F[2], &faces) || !mul_ok(faces, nv, &felems))
        return FVF_ERR_SIZE;
    if (elems == 0) return FVF_OK;
    if (!flux || !inv_d || !rhs) return FVF_ERR_NULL;
    const uint64_t esize = fp32 ? 4 : 8;
    if ((uintptr_t)flux % esize || (uintptr_t)inv_d % esize || (uintptr_t)rhs % esize)
        return FVF_ERR_ALIGN;
    const uint64_t rbytes = (uint64_t)elems * esize, fbytes = (uint64_t)felems * esize;
    const uint64_t wbytes = (uint64_t)n[dir] * esize;
    int st = check_device_array(flux, fbytes);
    if (st == FVF_OK) st = check_device_array(inv_d, wbytes);
    if (st == FVF_OK) st = check_device_array(rhs, rbytes);
    if (st != FVF_OK) return st;
    if (overlaps(rhs, rbytes, flux, fbytes) || overlaps(rhs, rbytes, inv_d, wbytes))
        return FVF_ERR_ALIAS;
    uint64_t launched = 0;
    const cudaError_t e = launch_advect_rhs(flux, inv_d, nv, n, dir, accumulate, fp32, rhs,
                                            (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API int advect_rhs(const double *flux, const double *inv_d, int nv, const int64_t extents[3],
                       int dir, double *rhs, void *stream) {
    return advect_rhs_impl(flux, inv_d, nv, extents, dir, false, false, rhs, stream);
}

FVF_API int advect_rhs_add(const double *flux, const double *inv_d, int nv,
                           const int64_t extents[3], int dir, double *rhs, void *stream) {
    return advect_rhs_impl(flux, inv_d, nv, extents, dir, true, false, rhs, stream);
}

FVF_API int advect_rhs_f32(const float *flux, const float *inv_d, int nv,
                           const int64_t extents[3], int dir, float *rhs, void *stream) {
    return advect_rhs_impl(flux, inv_d, nv, extents, dir, false, true, rhs, stream);
}

FVF_API int advect_rhs_add_f32(const float *flux, const float *inv_d, int nv,
                               const int64_t extents[3], int dir, float *rhs, void *stream) {
    return advect_rhs_impl(flux, inv_d, nv, extents, dir, true, true, rhs, stream);
}

// The inverse of the pack's axis exchange is the same exchange, so the copy
// back to the physical frame is the pack of the sweep-frame face box (its
// extents as the interior, ghost width 0), with the variables' planes of the
// one input array as the field table.
FVF_API int flux_unpack(const double *sweep_flux, int nv, const int64_t extents[3], int dir,
                        double *out, void *stream) {
    if (!extents) return FVF_ERR_NULL;
    if (dir < 0 || dir > 2) return FVF_ERR_DIR;
    if (nv < 0 || nv > FVF_MAX_NV) return FVF_ERR_NV;
    for (int a = 0; a < 3; ++a)
        if (extents[a] < 0) return FVF_ERR_SIZE;
    const int64_t n1 = extents[0], n2 = extents[1], n3 = extents[2];
    const int64_t S[3][3] = {{n1 + 1, n2, n3}, {n2 + 1, n1, n3}, {n3 + 1, n2, n1}};
    Box box;
    for (int a = 0; a < 3; ++a) {
        box.n[a] = S[dir][a];
        box.N[a] = S[dir][a];
        box.g[a] = 0;
    }
    int64_t t = 0, plane = 0, elems = 0;
    if (!mul_ok(box.n[0], box.n[1], &t) || !mul_ok(t, box.n[2], &plane) ||
        !mul_ok(plane, nv, &elems))
        return FVF_ERR_SIZE;
    if (n1 == 0 || n2 == 0 || n3 == 0 || elems == 0) return FVF_OK;
    if (!sweep_flux || !out) return FVF_ERR_NULL;
    if ((uintptr_t)sweep_flux % 8 || (uintptr_t)out % 8) return FVF_ERR_ALIGN;
    const uint64_t bytes = (uint64_t)elems * 8;
    int st = check_device_array(sweep_flux, bytes);
    if (st == FVF_OK) st = check_device_array(out, bytes);
    if (st != FVF_OK) return st;
    if (overlaps(sweep_flux, bytes, out, bytes)) return FVF_ERR_ALIAS;
    FieldTable table;
    std::memset(&table, 0, sizeof(table));
    for (int i = 0; i < nv; ++i) table.p[i] = sweep_flux + (int64_t)i * plane;
    uint64_t launched = 0;
    const cudaError_t e =
        launch_weno_pack(table, nv, box, dir, out, false, (cudaStream_t)stream, &launched);
    g_launches += launched;
    return cuda_status(e);
}

FVF_API const char *fvf_status_string(int status) {
    switch (status) {
        case FVF_OK: return "ok";
        case FVF_ERR_NULL: return "null pointer";
        case FVF_ERR_SIZE: return "invalid size";
        case FVF_ERR_DTYPE: return "invalid dtype";
        case FVF_ERR_DIR: return "invalid direction";
        case FVF_ERR_NV: return "invalid number of variables";
        case FVF_ERR_ALIAS: return "output overlaps an input";
        case FVF_ERR_ALPHA: return "alpha or a stage coefficient is not finite";
        case FVF_ERR_ALIGN: return "misaligned pointer";
        case FVF_ERR_NOT_DEVICE: return "pointer is not device memory of the current device";
        case FVF_ERR_RANGE: return "array runs past the end of its allocation";
        case FVF_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

FVF_API int fvf_last_cuda_error(void) { return g_last_cuda_error; }

FVF_API int fvf_device_error(int *flag) {
    if (!flag) return FVF_ERR_NULL;
    *flag = 0;
    int waits = 0, bounds = 0, b = 0;
    cudaError_t e = read_device_error(&waits);
    cudaError_t (*const readers[])(int *) = {read_bounds_diffuse2d, read_bounds_diffuse3d,
                                             read_bounds_pack, read_bounds_rhs, read_bounds_rk};
    for (auto rd : readers) {
        if (e != cudaSuccess) break;
        e = rd(&b);
        bounds |= b;
    }
    if (e != cudaSuccess) return cuda_status(e);
    *flag = ((waits & 1) ? 1 : 0) | (bounds ? 2 : 0) | ((waits & 2) ? 4 : 0);
    return FVF_OK;
}

FVF_API uint64_t fvf_launch_count(void) { return g_launches.load(); }
