// diffuse2d.cu -- explicit 2D 5-point diffusion step (FP32 and FP64) with
// ping-pong buffers, for sm_103a.
//
// Operation (Qiita, "Fortran 2018 GPU acceleration, part 3", section 3 and
// section 5.1): for interior cells
//     dst(i,j) = c + alpha*((((W + E) + S) + N) - 4c)
// and dst = 0 on the four edges, with the field column-major (i contiguous,
// section 4).  Every operation is rounded to nearest even on its own, in the
// order written: the round-to-nearest intrinsics below are never contracted
// into fused multiply-adds.  The single fused operation used, fma(-4, c, s),
// rounds the exact value s - 4c once, which is what s - fl(4c) gives whenever
// 4c is representable (4c is a power-of-two scaling, exact unless it
// overflows); cells with |c| >= 2^126 (FP32) or 2^1022 (FP64) take the
// two-operation form instead, so the result is bit-identical for every
// input.
//
// Thread mapping: the contiguous index i runs along the lanes of a warp, so
// every row access of a warp is one coalesced segment; one thread updates one
// cell (the spatial loops are the parallel ones, as the MFC pull request
// #2087 recommends for per-cell sweeps).
#include "fvf_internal.cuh"

namespace fvf {
namespace {

template <typename T>
struct Rn;

template <>
struct Rn<double> {
    static __device__ __forceinline__ double add(double a, double b) { return __dadd_rn(a, b); }
    static __device__ __forceinline__ double mul(double a, double b) { return __dmul_rn(a, b); }
    // s - 4c rounded once.
    static __device__ __forceinline__ double sub4(double s, double c) {
        if ((__double2hiint(c) & 0x7ff00000) >= 0x7fd00000)  // |c| >= 2^1022, NaN, Inf
            return __dsub_rn(s, __dmul_rn(4.0, c));
        return __fma_rn(-4.0, c, s);
    }
};

template <>
struct Rn<float> {
    static __device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
    static __device__ __forceinline__ float sub4(float s, float c) {
        if ((__float_as_uint(c) & 0x7f800000u) >= 0x7e800000u)  // |c| >= 2^126, NaN, Inf
            return __fsub_rn(s, __fmul_rn(4.0f, c));
        return __fmaf_rn(-4.0f, c, s);
    }
};

template <typename T>
__device__ __forceinline__ T update(T c, T w, T e, T s, T n, T alpha) {
    using R = Rn<T>;
    const T sum = R::add(R::add(R::add(w, e), s), n);
    return R::add(c, R::mul(alpha, R::sub4(sum, c)));
}

constexpr int kBx = 64;  // threads along i
constexpr int kBy = 4;   // threads along j

template <typename T>
__global__ void __launch_bounds__(kBx * kBy)
diffuse_step_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t nx, int64_t ny,
                    T alpha) {
    const int64_t i = (int64_t)blockIdx.x * kBx + threadIdx.x;
    if (i >= nx) return;
    for (int64_t j = (int64_t)blockIdx.y * kBy + threadIdx.y; j < ny;
         j += (int64_t)gridDim.y * kBy) {
        const int64_t c = i + nx * j;
        if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1) {
            dst[c] = T(0);
        } else {
            dst[c] = update<T>(src[c], src[c - 1], src[c + 1], src[c - nx], src[c + nx], alpha);
        }
    }
}

template <typename T>
cudaError_t run(T *u, T *v, int64_t nx, int64_t ny, T alpha, int64_t nsteps,
                cudaStream_t stream, uint64_t *launches) {
    const dim3 block(kBx, kBy);
    const int64_t gy = (ny + kBy - 1) / kBy;
    const dim3 grid((unsigned)((nx + kBx - 1) / kBx), (unsigned)(gy < 65535 ? gy : 65535));
    for (int64_t s = 1; s <= nsteps; ++s) {
        const T *src = (s & 1) ? u : v;
        T *dst = (s & 1) ? v : u;
        diffuse_step_kernel<T><<<grid, block, 0, stream>>>(src, dst, nx, ny, alpha);
        ++*launches;
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_diffuse2d(void *u, void *v, int64_t nx, int64_t ny, double alpha,
                             int64_t nsteps, bool fp64, cudaStream_t stream,
                             uint64_t *launches) {
    if (nx > (int64_t)kBx * 0x7fffffff) return cudaErrorInvalidValue;
    if (fp64)
        return run<double>(static_cast<double *>(u), static_cast<double *>(v), nx, ny, alpha,
                           nsteps, stream, launches);
    return run<float>(static_cast<float *>(u), static_cast<float *>(v), nx, ny, (float)alpha,
                      nsteps, stream, launches);
}

}  // namespace fvf
