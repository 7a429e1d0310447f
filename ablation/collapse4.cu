// collapse4.cu -- ablation kernels for the benchmark, not part of libfvf.
//
// MFlowCode/MFC pull request #2087 ("Summary", "Why this is faster") replaces
// loops that give every (variable, cell) pair its own GPU iteration -- the
// "collapse=4" mapping, where each thread decomposes a flat index into
// (j, k, l, i) and, in the flux difference, loads the inverse spacing per
// element -- with one thread per cell looping over the variables.  libfvf
// implements the second form.  This file implements the first for two of the
// sweeps (the x pack and the x flux difference), with the same arithmetic,
// so that the benchmark can time the two mappings against each other on
// GB300.  Built into libfvf_ablation.so by buildlib.build_ablation().
#include <cuda_runtime.h>
#include <stdint.h>

#define ABL_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kMaxNv = 64;
constexpr int kThreads = 256;

struct Table {
    const double *p[kMaxNv];
};

// out(a, b, c, i) = f_i(a, b+g2, c+g3), one thread per output element.
__global__ void __launch_bounds__(kThreads)
pack_x_collapse4_kernel(Table t, int64_t total, int64_t M1, int64_t n2, int64_t n3, int64_t N1,
                        int64_t N2, int64_t g2, int64_t g3, double *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += stride) {
        const int64_t a = e % M1;
        int64_t r = e / M1;
        const int64_t b = r % n2;
        r /= n2;
        const int64_t c = r % n3;
        const int64_t i = r / n3;
        out[e] = __ldg(t.p[i] + a + N1 * ((b + g2) + N2 * (c + g3)));
    }
}

// rhs(j,k,l,i) = inv_d(j) * (F(j-1,k,l,i) - F(j,k,l,i)), one thread per
// (cell, variable) element, inv_d loaded for every element.
__global__ void __launch_bounds__(kThreads)
rhs_x_collapse4_kernel(const double *__restrict__ flux, const double *__restrict__ inv_d,
                       int64_t total, int64_t n1, int64_t n2, int64_t n3,
                       double *__restrict__ rhs) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += stride) {
        const int64_t j = e % n1;
        int64_t r = e / n1;
        const int64_t k = r % n2;
        r /= n2;
        const int64_t l = r % n3;
        const int64_t i = r / n3;
        const int64_t lo = j + (n1 + 1) * (k + n2 * (l + n3 * i));
        rhs[e] = __dmul_rn(__ldg(inv_d + j), __dsub_rn(__ldg(flux + lo), __ldg(flux + lo + 1)));
    }
}

unsigned grid_for(int64_t total) {
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    return (unsigned)(blocks < 0x7fffffff ? blocks : 0x7fffffff);
}

}  // namespace

// Both entry points take device pointers and enqueue one launch on `stream`;
// they return 0, 1 for a bad argument, or 2 for a failed launch.  The layouts
// are those of weno_pack (dir 0) and advect_rhs (dir 0) in include/fvf.h.
ABL_API int ablation_pack_x_collapse4(const double *const *fields, int nv,
                                      const int64_t extents[3], int ghost, double *out,
                                      void *stream) {
    if (!fields || !extents || !out || nv < 1 || nv > kMaxNv || ghost < 0) return 1;
    const int64_t n1 = extents[0], n2 = extents[1], n3 = extents[2];
    if (n1 < 1 || n2 < 1 || n3 < 1) return 1;
    const int64_t g = ghost;
    const int64_t N1 = n1 > 1 ? n1 + 2 * g : 1, N2 = n2 > 1 ? n2 + 2 * g : 1;
    const int64_t g2 = n2 > 1 ? g : 0, g3 = n3 > 1 ? g : 0;
    Table t;
    for (int i = 0; i < kMaxNv; ++i) t.p[i] = i < nv ? fields[i] : nullptr;
    const int64_t total = N1 * n2 * n3 * nv;
    pack_x_collapse4_kernel<<<grid_for(total), kThreads, 0, (cudaStream_t)stream>>>(
        t, total, N1, n2, n3, N1, N2, g2, g3, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

ABL_API int ablation_rhs_x_collapse4(const double *flux, const double *inv_d, int nv,
                                     const int64_t extents[3], double *rhs, void *stream) {
    if (!flux || !inv_d || !extents || !rhs || nv < 1) return 1;
    const int64_t n1 = extents[0], n2 = extents[1], n3 = extents[2];
    if (n1 < 1 || n2 < 1 || n3 < 1) return 1;
    const int64_t total = n1 * n2 * n3 * nv;
    rhs_x_collapse4_kernel<<<grid_for(total), kThreads, 0, (cudaStream_t)stream>>>(
        flux, inv_d, total, n1, n2, n3, rhs);
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
