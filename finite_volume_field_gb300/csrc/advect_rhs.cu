// advect_rhs.cu -- finite-volume flux-difference source for sm_103a,
// assigned or accumulated into an existing rhs.
//
// Operation (MFlowCode/MFC pull request #2087, "Changes",
// s_compute_advection_source_term, x/y/z flux differences):
//     rhs(j,k,l,i) = inv_d(c) * (F(c-1) - F(c))
// along the swept axis c, one subtraction then one multiplication, each
// rounded to nearest even (round-to-nearest intrinsics, never contracted), in
// binary64 or, for the FP32 entry points, binary32.
// Two FP64 operations per element would keep this kernel on GB300's FP64
// unit, well below the HBM roof.  The multiplication by inv_d runs on the
// integer pipes instead (fp64_emu.cuh: an exact binary64 product, the factor
// prepared once per cell) for three of every four variables (kMulMask = 7,
// one bit per slot of a load batch); on GB300 this measured 20-26% faster
// than all-FP64 and than emulating all four (the integer pipes saturate
// then).  The accumulating form takes all four (kMulMaskAcc).  Moving the
// subtraction instead measured slower: the exact addition costs about twice
// the integer instructions of the product.
//
// Mapping ("Why this is faster" on the same page): one thread per spatial
// cell; the inverse spacing is loaded once per cell, outside the variable
// loop, and the face offsets are computed once and reused for every variable.
// The contiguous index j is on the lanes, so every load and store of a warp
// is coalesced in all three directions.
#include "fp64_emu.cuh"
#include "fvf_internal.cuh"

namespace fvf {
namespace {

// Variable slots of a load batch whose product runs on the integer pipes
// (bit q: slot q): three of four for the assigning form; all four for the
// accumulating form, whose extra read and add change the balance (2-7%
// faster there).
constexpr int kMulMask = 7;
constexpr int kMulMaskAcc = 15;

// Threads per block, per form, as measured on GB300 at 8 x 201^3 and
// 4800 x 1200 x 7 (one box, back to back): the assigning FP64 form at 128
// (2-3.5% faster than 256 in every direction; 64 is slower in y), the
// accumulating FP64 form at 64 (2-10% faster than 256, 1-2% than 128), the
// FP32 form at 256 (within 1% of 64 and 128).
template <bool ACC, typename T>
__host__ __device__ constexpr int threads_of() {
    return sizeof(T) == 4 ? 256 : (ACC ? 64 : 128);
}

// Minimum resident blocks per SM, per form (a register cap; 0 = none), as
// measured on GB300 at 8 x 201^3 and 4800 x 1200 x 7: the FP32 form at 6
// blocks of 256 threads (more loads in flight for 4-byte elements: 0.099 ms
// at 4 blocks, 0.093 ms at 6, 0.146 ms at 8, timed back to back); the
// assigning FP64 y form at 12 blocks of 128 threads (0.121 / 0.179 ms for
// the 2D / 3D y sweeps, against 0.127 / 0.186 with no cap and 0.129-0.133 /
// 0.189-0.193 with 8 or 10).  The other FP64 forms take none: with 256-thread
// blocks a cap on x and z measured 5-13% slower, and on the accumulating y
// form (64-thread blocks) a minimum of 20 blocks measured 0.182 / 0.286 ms
// against 0.168 / 0.265 with none.
template <int DIR, bool ACC, typename T>
constexpr int min_blocks() {
    return sizeof(T) == 4 ? 6 : (DIR == 1 && !ACC ? 12 : 0);
}

// variables per load batch: 4 FP64 or 8 FP32, 64 bytes of face loads each
template <typename T>
__host__ __device__ constexpr int group_of() { return sizeof(T) == 4 ? 8 : 4; }

// Face difference F(c-1) - F(c) on the FP64 unit.
template <int Q>
__device__ __forceinline__ double face_diff(double lo, double hi) { return __dsub_rn(lo, hi); }

// FP32 form: binary32 operations, each rounded to nearest even.
template <int Q>
__device__ __forceinline__ float face_diff(float lo, float hi) { return __fsub_rn(lo, hi); }
// inv_d(c) times a face difference: on the FP64 unit, or on the integer
// pipes (fp64_emu.cuh, the factor prepared once per cell) for the variable
// slots whose bit is set in MASK.
template <typename T>
struct Scale;

template <>
struct Scale<double> {
    double w;
    emu::MulConst m;
    __device__ explicit Scale(double w_) : w(w_), m(emu::mul_const(w_)) {}
    template <int MASK, int Q>
    __device__ __forceinline__ double apply(double d) const {
        if ((MASK >> Q) & 1) return emu::from_bits(emu::mul_const_bits(emu::bits(d), m));
        return __dmul_rn(w, d);
    }
};

template <>
struct Scale<float> {
    float w;
    __device__ explicit Scale(float w_) : w(w_) {}
    template <int MASK, int Q>
    __device__ __forceinline__ float apply(float d) const { return __fmul_rn(w, d); }
};
__device__ __forceinline__ double add_rn(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }

// F extents per variable (F1, F2, F3); the high face of a cell is `step`
// elements after its low face (1, F1 or F1*F2).  One thread per cell (j, k)
// of a plane l, the (j, k) pairs flattened over the block so that every lane
// has a cell whatever n1 is: the kernel is bound by the FP64 unit, which
// charges idle lanes.
template <int DIR, bool ACC, typename Idx, typename Off, typename T>
__global__ void __launch_bounds__(threads_of<ACC, T>(), min_blocks<DIR, ACC, T>())
advect_rhs_kernel(const T *__restrict__ flux, const T *__restrict__ inv_d, int nv,
                  int64_t n1_, int64_t n2_, int64_t n3_, T *__restrict__ rhs) {
    const Idx n1 = (Idx)n1_, n2 = (Idx)n2_;
    const Idx plane = n1 * n2;
    const Idx jk = (Idx)blockIdx.x * threads_of<ACC, T>() + threadIdx.x;
    if (jk >= plane) return;
    const Idx k = jk / n1, j = jk - k * n1;
    // flat offsets in Off: 32-bit when every element index of both arrays
    // fits (the launcher checks), else 64-bit
    const Off n3 = (Off)n3_;
    const Off F1 = DIR == 0 ? (Off)n1 + 1 : (Off)n1;
    const Off F2 = DIR == 1 ? (Off)n2 + 1 : (Off)n2;
    const Off F3 = DIR == 2 ? n3 + 1 : n3;
    const Off fplane = F1 * F2 * F3;
    const Off rplane = (Off)plane * n3;
    const Off step = DIR == 0 ? 1 : (DIR == 1 ? F1 : F1 * F2);
    const Off nw = DIR == 0 ? (Off)n1 : (DIR == 1 ? (Off)n2 : n3);  // inv_d extent
    const Off fall = fplane * nv, rall = rplane * nv;  // flux and rhs extents
    (void)nw; (void)fall; (void)rall;
    const T wjk = DIR == 0 ? (FVF_IN(j, nw) ? __ldg(inv_d + j) : T(0))
                           : (DIR == 1 ? (FVF_IN(k, nw) ? __ldg(inv_d + k) : T(0)) : T(0));
    for (Off l = blockIdx.y; l < n3; l += gridDim.y) {
        const Scale<T> w(DIR == 2 ? (FVF_IN(l, nw) ? __ldg(inv_d + l) : T(0)) : wjk);
        const Off lo = (Off)j + F1 * ((Off)k + F2 * l);  // face c-1 at position c
        const Off ro = (Off)jk + (Off)plane * l;
        const T *f = flux + lo;
        T *r = rhs + ro;
        constexpr int kGroup = group_of<T>();
        constexpr int kMask = ACC ? kMulMaskAcc : kMulMask;
        for (int i0 = 0; i0 < nv; i0 += kGroup) {
            T a[kGroup], b[kGroup], old[kGroup];
#pragma unroll
            for (int q = 0; q < kGroup; ++q) {
                if (i0 + q < nv) {
                    const Off fo = (Off)(i0 + q) * fplane;
                    a[q] = FVF_IN(lo + fo, fall) ? __ldg(f + fo) : T(0);
                    b[q] = FVF_IN(lo + fo + step, fall) ? __ldg(f + fo + step) : T(0);
                    if (ACC)
                        old[q] = FVF_IN(ro + (Off)(i0 + q) * rplane, rall)
                                     ? r[(Off)(i0 + q) * rplane] : T(0);
                }
            }
#define FVF_RHS_Q(Q)                                                                    \
    if (Q < kGroup && i0 + Q < nv) {                                                    \
        const T term = w.template apply<kMask, Q>(face_diff<Q>(a[Q], b[Q]));        \
        /* accumulate form: the term added once to the existing rhs */                 \
        if (FVF_IN(ro + (Off)(i0 + Q) * rplane, rall))                                  \
            r[(Off)(i0 + Q) * rplane] = ACC ? add_rn(old[Q], term) : term;             \
    }
            FVF_RHS_Q(0)
            FVF_RHS_Q(1)
            FVF_RHS_Q(2)
            FVF_RHS_Q(3)
            FVF_RHS_Q(4)
            FVF_RHS_Q(5)
            FVF_RHS_Q(6)
            FVF_RHS_Q(7)
            FVF_RHS_Q(8)
            FVF_RHS_Q(9)
            FVF_RHS_Q(10)
            FVF_RHS_Q(11)
            FVF_RHS_Q(12)
            FVF_RHS_Q(13)
            FVF_RHS_Q(14)
            FVF_RHS_Q(15)
#undef FVF_RHS_Q
        }
    }
}

// Which forms take 32-bit flat offsets, as measured on GB300 at 8 x 201^3:
// the FP32 form (3-20% faster), the FP64 z forms and the assigning FP64 y
// form (2-3% faster); the other FP64 forms measured 1-16% slower, the
// compiler's register allocation of the emulated products differing.
template <int DIR, bool ACC, typename T>
constexpr bool off32() {
    return sizeof(T) == 4 || DIR == 2 || (DIR == 1 && !ACC);
}

template <int DIR, bool ACC, typename T>
void launch_typed(const T *flux, const T *inv_d, int nv, const int64_t n[3], T *rhs,
                  cudaStream_t stream) {
    const int64_t plane = n[0] * n[1];
    constexpr int kThreads = threads_of<ACC, T>();
    const dim3 grid((unsigned)((plane + kThreads - 1) / kThreads),
                    (unsigned)(n[2] < 65535 ? n[2] : 65535));
    // 32-bit (j, k) arithmetic while the plane index fits, and, for the
    // forms where off32<>() says so, 32-bit flat offsets too while every flux
    // and rhs element index fits (the flux array, one face layer larger
    // along the swept axis, is the larger)
    const int64_t lim = (int64_t)1 << 31;
    const int64_t fall = (n[0] + 1) * (n[1] + 1) * (n[2] + 1) * nv;
    if (off32<DIR, ACC, T>() && fall + plane + kThreads < lim)
        advect_rhs_kernel<DIR, ACC, uint32_t, uint32_t, T><<<grid, kThreads, 0, stream>>>(
            flux, inv_d, nv, n[0], n[1], n[2], rhs);
    else if (plane + kThreads < lim)
        advect_rhs_kernel<DIR, ACC, uint32_t, int64_t, T><<<grid, kThreads, 0, stream>>>(
            flux, inv_d, nv, n[0], n[1], n[2], rhs);
    else
        advect_rhs_kernel<DIR, ACC, int64_t, int64_t, T><<<grid, kThreads, 0, stream>>>(
            flux, inv_d, nv, n[0], n[1], n[2], rhs);
}

template <typename T>
void launch_dir(const T *flux, const T *inv_d, int nv, const int64_t n[3], int dir,
                bool accumulate, T *rhs, cudaStream_t stream) {
    if (dir == 0) {
        if (accumulate) launch_typed<0, true>(flux, inv_d, nv, n, rhs, stream);
        else launch_typed<0, false>(flux, inv_d, nv, n, rhs, stream);
    } else if (dir == 1) {
        if (accumulate) launch_typed<1, true>(flux, inv_d, nv, n, rhs, stream);
        else launch_typed<1, false>(flux, inv_d, nv, n, rhs, stream);
    } else {
        if (accumulate) launch_typed<2, true>(flux, inv_d, nv, n, rhs, stream);
        else launch_typed<2, false>(flux, inv_d, nv, n, rhs, stream);
    }
}

}  // namespace

FVF_BOUNDS_READER(read_bounds_rhs)

cudaError_t launch_advect_rhs(const void *flux, const void *inv_d, int nv, const int64_t n[3],
                              int dir, bool accumulate, bool fp32, void *rhs,
                              cudaStream_t stream, uint64_t *launches) {
    // the smallest block (64 threads) gives the largest grid
    const int64_t gx = (n[0] * n[1] + 63) / 64;
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    if (fp32)
        launch_dir<float>(static_cast<const float *>(flux), static_cast<const float *>(inv_d), nv,
                          n, dir, accumulate, static_cast<float *>(rhs), stream);
    else
        launch_dir<double>(static_cast<const double *>(flux), static_cast<const double *>(inv_d),
                           nv, n, dir, accumulate, static_cast<double *>(rhs), stream);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace fvf
