// rk_stage.cu -- SSPRK3 stage update for sm_103a, alone (given rhs) and
// fused with the finite-volume flux difference.
//
// Operation (Mallard documentation, "Design: single-GPU performance and
// parallel scaling": "Hardware and method", a step is three SSPRK3 stages;
// "Baseline (main)", the per-stage rhs and axpby kernels), per cell c and
// variable i:
//     rhs = inv_x(j)*(Fx(j-1) - Fx(j)) [+ inv_y(k)*(Fy(k-1) - Fy(k))]
//                                      [+ inv_z(l)*(Fz(l-1) - Fz(l))]
//     t   = u + dt*rhs
//     out = a*u0 + b*t
// every operation rounded to nearest even in this order (the flux terms as
// in the x/y/z flux differences of MFlowCode/MFC pull request #2087,
// "Changes", s_compute_advection_source_term).  The fused kernel keeps rhs
// in registers: per element it reads u0, u and the faces and writes out, in
// place of the flux difference writing rhs and the update reading it back.
//
// Mapping: one thread per cell (j, k) of a plane l, the (j, k) pairs
// flattened so that every lane of every warp has a cell (the rows of 201
// cells would leave a fifth of the lanes of a row-per-block mapping idle, and
// the kernel is bound by the FP64 unit, which charges idle lanes).  The
// variables are processed in chunks of kChunk inside the thread: the chunk's
// loads are all issued before its stores, since out may be u or u0 itself
// and the compiler must not assume that it is not.
//
// FP64 throughput.  The fused 3D update is 13 FP64 operations per element
// against 48 bytes of HBM traffic, far above GB300's FP64-to-bandwidth
// ratio.  Its six multiplications run on the integer pipes instead, as exact
// binary64 products by factors prepared once (fp64_emu.cuh: the x/y/z
// inverse spacings, dt, a and b), leaving the seven additions on the FP64
// unit.  With one variable per load batch this measured fastest on GB300, 36%
// below the all-FP64 kernel (the update alone measured fastest with one
// variable per batch as well).  Additions on the integer pipes as well (the
// y and z terms, u + dt*rhs, the final sum, the face differences, any
// choice of them) measured slower: an exact addition costs about twice the
// integer instructions of a product.
#include "fp64_emu.cuh"
#include "fvf_internal.cuh"

namespace fvf {
namespace {

// Threads per block: 128.  Per call on 8 x 201^3 on GB300 (one box, back
// to back): the stage fused with the x, y and z flux differences 0.937 ms
// against 0.965 with 256 threads (0.935 with 64); fused with x alone 0.581
// against 0.594 (0.595 with 64); the update alone 0.429 with 128 or 256
// (0.445 with 64).
constexpr int kThreads = 128;
constexpr int kChunk = 1;   // variables per load batch

__device__ __forceinline__ double add_rn(double x, double y) { return __dadd_rn(x, y); }
__device__ __forceinline__ double sub_rn(double x, double y) { return __dsub_rn(x, y); }

// w * x on the integer pipes, the factor w prepared in m (fp64_emu.cuh)
__device__ __forceinline__ double mul_rn(const emu::MulConst &m, double x) {
    return emu::from_bits(emu::mul_const_bits(emu::bits(x), m));
}

template <bool FUSED, bool FY, bool FZ, typename Idx>
__global__ void __launch_bounds__(kThreads)
rk_stage_kernel(RkStageArgs A) {
    const Idx n1 = (Idx)A.n[0], n2 = (Idx)A.n[1];
    const Idx plane_jk = n1 * n2;
    const Idx jk = (Idx)blockIdx.x * kThreads + threadIdx.x;
    if (jk >= plane_jk) return;
    const Idx k = jk / n1, j = jk - k * n1;
    const int64_t n3 = A.n[2];
    const int64_t cplane = (int64_t)plane_jk * n3;  // cells per variable
    const int64_t fxp = (int64_t)(n1 + 1) * n2 * n3, fyp = (int64_t)n1 * (n2 + 1) * n3,
                  fzp = (int64_t)plane_jk * (n3 + 1);
    const int64_t call = cplane * A.nv;  // extents of the cell and face arrays
    const int64_t xall = (FUSED ? fxp : cplane) * A.nv, yall = fyp * A.nv, zall = fzp * A.nv;
    (void)call; (void)xall; (void)yall; (void)zall;
    const double wx = FUSED && FVF_IN(j, n1) ? __ldg(A.w[0] + j) : 0.0;
    const double wy = FY && FVF_IN(k, n2) ? __ldg(A.w[1] + k) : 0.0;
    const emu::MulConst mx = emu::mul_const(wx), my = emu::mul_const(wy);
    const emu::MulConst mdt = emu::mul_const(A.dt), ma = emu::mul_const(A.a),
                        mb = emu::mul_const(A.b);
    for (int64_t l = blockIdx.y; l < n3; l += gridDim.y) {
        const double wz = FZ && FVF_IN(l, n3) ? __ldg(A.w[2] + l) : 0.0;
        const emu::MulConst mz = emu::mul_const(wz);
        const int64_t c = (int64_t)jk + (int64_t)plane_jk * l;
        const int64_t xlo = (int64_t)j + (int64_t)(n1 + 1) * ((int64_t)k + (int64_t)n2 * l);
        const int64_t ylo = (int64_t)j + (int64_t)n1 * ((int64_t)k + (int64_t)(n2 + 1) * l);
        const int64_t zlo = c;
        for (int i0 = 0; i0 < A.nv; i0 += kChunk) {
            double u0v[kChunk], uv[kChunk], r[kChunk];
            double xl[kChunk], xh[kChunk], yl[kChunk], yh[kChunk], zl[kChunk], zh[kChunk];
#pragma unroll
            for (int q = 0; q < kChunk; ++q) {
                if (i0 + q < A.nv) {
                    const int64_t iv = i0 + q;
                    const bool cin = FVF_IN(c + iv * cplane, call);
                    u0v[q] = cin ? A.u0[c + iv * cplane] : 0.0;
                    uv[q] = cin ? A.u[c + iv * cplane] : 0.0;
                    if (FUSED) {
                        const bool in = FVF_IN(xlo + iv * fxp + 1, xall);
                        xl[q] = in ? __ldg(A.f[0] + xlo + iv * fxp) : 0.0;
                        xh[q] = in ? __ldg(A.f[0] + xlo + iv * fxp + 1) : 0.0;
                    } else {
                        r[q] = cin ? __ldg(A.f[0] + c + iv * cplane) : 0.0;
                    }
                    if (FY) {
                        const bool in = FVF_IN(ylo + iv * fyp + n1, yall);
                        yl[q] = in ? __ldg(A.f[1] + ylo + iv * fyp) : 0.0;
                        yh[q] = in ? __ldg(A.f[1] + ylo + iv * fyp + n1) : 0.0;
                    }
                    if (FZ) {
                        const bool in = FVF_IN(zlo + iv * fzp + plane_jk, zall);
                        zl[q] = in ? __ldg(A.f[2] + zlo + iv * fzp) : 0.0;
                        zh[q] = in ? __ldg(A.f[2] + zlo + iv * fzp + plane_jk) : 0.0;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kChunk; ++q) {
                if (i0 + q < A.nv) {
                    const int v = i0 + q;
                    double rr;
                    if (FUSED) {
                        rr = mul_rn(mx, sub_rn(xl[q], xh[q]));
                        if (FY) rr = add_rn(rr, mul_rn(my, sub_rn(yl[q], yh[q])));
                        if (FZ) rr = add_rn(rr, mul_rn(mz, sub_rn(zl[q], zh[q])));
                    } else {
                        rr = r[q];
                    }
                    const double t = add_rn(uv[q], mul_rn(mdt, rr));
                    if (FVF_IN(c + (int64_t)v * cplane, call))
                        A.out[c + (int64_t)v * cplane] =
                            add_rn(mul_rn(ma, u0v[q]), mul_rn(mb, t));
                }
            }
        }
    }
}

template <bool FUSED, bool FY, bool FZ>
cudaError_t launch_typed(const RkStageArgs &A, cudaStream_t stream) {
    const int64_t plane = A.n[0] * A.n[1];
    const int64_t gx = (plane + kThreads - 1) / kThreads;
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)(A.n[2] < 65535 ? A.n[2] : 65535));
    // 32-bit (j, k) arithmetic while the plane index and n1 + 1 fit
    if (plane + A.n[0] + kThreads < ((int64_t)1 << 31))
        rk_stage_kernel<FUSED, FY, FZ, uint32_t><<<grid, kThreads, 0, stream>>>(A);
    else
        rk_stage_kernel<FUSED, FY, FZ, int64_t><<<grid, kThreads, 0, stream>>>(A);
    return cudaSuccess;
}

}  // namespace

FVF_BOUNDS_READER(read_bounds_rk)

cudaError_t launch_rk_stage(const RkStageArgs &A, bool fused, cudaStream_t stream,
                            uint64_t *launches) {
    cudaError_t e;
    if (!fused) {
        e = launch_typed<false, false, false>(A, stream);
    } else {
        const bool fy = A.f[1] != nullptr, fz = A.f[2] != nullptr;
        if (fy && fz) e = launch_typed<true, true, true>(A, stream);
        else if (fy) e = launch_typed<true, true, false>(A, stream);
        else if (fz) e = launch_typed<true, false, true>(A, stream);
        else e = launch_typed<true, false, false>(A, stream);
    }
    if (e != cudaSuccess) return e;
    ++*launches;
    return cudaGetLastError();
}

}  // namespace fvf
