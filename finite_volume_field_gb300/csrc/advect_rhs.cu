// advect_rhs.cu -- finite-volume flux-difference source for sm_103a,
// assigned or accumulated into an existing rhs.
//
// Operation (MFlowCode/MFC pull request #2087, "Changes",
// s_compute_advection_source_term, x/y/z flux differences):
//     rhs(j,k,l,i) = inv_d(c) * (F(c-1) - F(c))
// along the swept axis c, one subtraction then one multiplication, each
// rounded to nearest even (round-to-nearest intrinsics, never contracted).
// Two FP64 operations per element keep this kernel on GB300's FP64 unit:
// moving the subtraction to the integer pipes (fp64_emu.cuh) was measured
// slower here (the integer ALU pipe saturates first), unlike in the
// diffusion update.
//
// Mapping ("Why this is faster" on the same page): one thread per spatial
// cell; the inverse spacing is loaded once per cell, outside the variable
// loop, and the face offsets are computed once and reused for every variable.
// The contiguous index j is on the lanes, so every load and store of a warp
// is coalesced in all three directions.
#include "fvf_internal.cuh"

namespace fvf {
namespace {

// F extents per variable (F1, F2, F3); the high face of a cell is `step`
// elements after its low face (1, F1 or F1*F2).
template <int DIR, bool ACC>
__global__ void __launch_bounds__(256)
advect_rhs_kernel(const double *__restrict__ flux, const double *__restrict__ inv_d, int nv,
                  int64_t n1, int64_t n2, int64_t n3, double *__restrict__ rhs) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n1) return;
    const int64_t F1 = DIR == 0 ? n1 + 1 : n1;
    const int64_t F2 = DIR == 1 ? n2 + 1 : n2;
    const int64_t F3 = DIR == 2 ? n3 + 1 : n3;
    const int64_t fplane = F1 * F2 * F3;
    const int64_t rplane = n1 * n2 * n3;
    const int64_t step = DIR == 0 ? 1 : (DIR == 1 ? F1 : F1 * F2);
    for (int64_t kl = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; kl < n2 * n3;
         kl += (int64_t)gridDim.y * blockDim.y) {
        const int64_t k = kl % n2, l = kl / n2;
        const double w = __ldg(inv_d + (DIR == 0 ? j : (DIR == 1 ? k : l)));
        const int64_t lo = j + F1 * (k + F2 * l);  // face c-1 sits at stored position c
        const double *f = flux + lo;
        double *r = rhs + j + n1 * kl;
#pragma unroll 4
        for (int i = 0; i < nv; ++i) {
            const double a = __ldg(f + (int64_t)i * fplane);
            const double b = __ldg(f + (int64_t)i * fplane + step);
            const double term = __dmul_rn(w, __dsub_rn(a, b));
            // accumulate form: the term added once to the existing rhs
            r[(int64_t)i * rplane] = ACC ? __dadd_rn(r[(int64_t)i * rplane], term) : term;
        }
    }
}

}  // namespace

cudaError_t launch_advect_rhs(const double *flux, const double *inv_d, int nv,
                              const int64_t n[3], int dir, bool accumulate, double *rhs,
                              cudaStream_t stream, uint64_t *launches) {
    const dim3 block(64, 4);
    const int64_t gx = (n[0] + 63) / 64;
    const int64_t gy = (n[1] * n[2] + 3) / 4;
    if (gx > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)(gy < 65535 ? gy : 65535));
#define FVF_RHS_LAUNCH(D, A) \
    advect_rhs_kernel<D, A><<<grid, block, 0, stream>>>(flux, inv_d, nv, n[0], n[1], n[2], rhs)
    if (dir == 0) {
        if (accumulate) FVF_RHS_LAUNCH(0, true); else FVF_RHS_LAUNCH(0, false);
    } else if (dir == 1) {
        if (accumulate) FVF_RHS_LAUNCH(1, true); else FVF_RHS_LAUNCH(1, false);
    } else {
        if (accumulate) FVF_RHS_LAUNCH(2, true); else FVF_RHS_LAUNCH(2, false);
    }
#undef FVF_RHS_LAUNCH
    ++*launches;
    return cudaGetLastError();
}

}  // namespace fvf
