// weno_pack.cu -- multi-variable WENO input pack for sm_103a.
//
// Operation (MFlowCode/MFC pull request #2087, "Changes",
// s_pack_weno_input_arr): out(a,b,c,i) = field_i(...) with the swept axis
// first (x: no permutation; y: j and k exchanged; z: j and l exchanged), the
// swept axis covering its ghost cells and the transverse axes their interior.
// A pure 64-bit copy.
//
// Mapping ("Why this is faster" on the same page): one thread per spatial
// output cell, the variable loop sequential inside the thread, the index
// arithmetic done once per cell and reused for every variable.  x keeps the
// contiguous index on the lanes for both the load and the store.  y and z are
// transposes: a block stages a 32 x 32 tile of each variable in shared memory
// so that both the global load (along j) and the global store (along the
// swept axis) are coalesced.
#include "fvf_internal.cuh"

namespace fvf {
namespace {

constexpr int kTile = 32;
constexpr int kRows = 8;  // threads along the second tile axis

// x: out(a, b, c, i) = f_i(a, b+g2, c+g3); (M1, M2, M3) = (N1, n2, n3).
__global__ void __launch_bounds__(256)
pack_x_kernel(FieldTable t, int nv, int64_t N1, int64_t N2, int64_t n2, int64_t n3,
              int64_t g2, int64_t g3, double *__restrict__ out) {
    const int64_t a = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= N1) return;
    const int64_t plane = N1 * n2 * n3;
    for (int64_t bc = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; bc < n2 * n3;
         bc += (int64_t)gridDim.y * blockDim.y) {
        const int64_t b = bc % n2, c = bc / n2;
        const int64_t src = a + N1 * ((b + g2) + N2 * (c + g3));
        double *o = out + a + N1 * bc;
#pragma unroll 8
        for (int i = 0; i < kMaxNv; ++i) {
            if (i >= nv) break;
            o[(int64_t)i * plane] = __ldg(t.p[i] + src);
        }
    }
}

// Transposing pack (y or z).  The tile spans the swept axis (output-fast,
// index a) and the j axis (input-fast, index jj); the third axis (index q) is
// fixed per block.
//   y: a = k (0..N2-1), jj = j (interior), q = l (interior); M = (N2, n1, n3)
//      src = (jj+g1) + N1*(a + N2*(q+g3)),  dst = a + N2*(jj + n1*q)
//   z: a = l (0..N3-1), jj = j (interior), q = k (interior); M = (N3, n2, n1)
//      src = (jj+g1) + N1*((q+g2) + N2*a),  dst = a + N3*(q + n2*jj)
// src = (jj + g1) + sa*a + sq*(q + gq); dst = a + da*jj + dq*q.
// The tile is double-buffered across variables: the loads of variable i+1
// are in flight while variable i is stored, with one barrier per variable.
constexpr int kPer = kTile / kRows;

__global__ void __launch_bounds__(kTile * kRows)
pack_transpose_kernel(FieldTable t, int nv, int64_t na, int64_t nj, int64_t nq, int64_t g1,
                      int64_t gq, int64_t sa, int64_t sq, int64_t da, int64_t dq,
                      int64_t plane, int64_t tiles_a, int64_t tiles_j,
                      double *__restrict__ out) {
    __shared__ double tile[2][kTile][kTile + 1];
    int64_t blk = blockIdx.x;
    const int64_t ta = blk % tiles_a;
    blk /= tiles_a;
    const int64_t tj = blk % tiles_j;
    const int64_t q = blk / tiles_j;
    const int64_t a0 = ta * kTile, j0 = tj * kTile;
    const int tx = threadIdx.x, ty = threadIdx.y;
    // load side: lanes along j (contiguous in the field), rows along a
    const int64_t jl = j0 + tx;
    const int64_t src0 = (jl + g1) + sa * (a0 + ty) + sq * (q + gq);
    bool lok[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) lok[r] = jl < nj && a0 + ty + r * kRows < na;
    // store side: lanes along a (contiguous in the output), rows along j
    const int64_t as = a0 + tx;
    const int64_t dst0 = as + da * (j0 + ty) + dq * q;
    bool sok[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) sok[r] = as < na && j0 + ty + r * kRows < nj;

    double v[kPer];
    {
        const double *f = t.p[0];
#pragma unroll
        for (int r = 0; r < kPer; ++r) v[r] = lok[r] ? __ldg(f + src0 + sa * (r * kRows)) : 0.0;
#pragma unroll
        for (int r = 0; r < kPer; ++r) tile[0][ty + r * kRows][tx] = v[r];
    }
    __syncthreads();
    for (int i = 0; i < nv; ++i) {
        const int buf = i & 1;
        const bool more = i + 1 < nv;
        if (more) {
            const double *f = t.p[i + 1];
#pragma unroll
            for (int r = 0; r < kPer; ++r)
                v[r] = lok[r] ? __ldg(f + src0 + sa * (r * kRows)) : 0.0;
        }
        double *o = out + (int64_t)i * plane + dst0;
#pragma unroll
        for (int r = 0; r < kPer; ++r)
            if (sok[r]) o[da * (r * kRows)] = tile[buf][tx][ty + r * kRows];
        if (more) {
#pragma unroll
            for (int r = 0; r < kPer; ++r) tile[buf ^ 1][ty + r * kRows][tx] = v[r];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_weno_pack(const FieldTable &fields, int nv, const Box &box, int dir,
                             double *out, cudaStream_t stream, uint64_t *launches) {
    const int64_t n1 = box.n[0], n2 = box.n[1], n3 = box.n[2];
    const int64_t N1 = box.N[0], N2 = box.N[1], N3 = box.N[2];
    const int64_t g1 = box.g[0], g2 = box.g[1], g3 = box.g[2];
    if (dir == 0) {
        const dim3 block(64, 4);
        const int64_t gx = (N1 + 63) / 64;
        const int64_t gy = (n2 * n3 + 3) / 4;
        if (gx > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)gx, (unsigned)(gy < 65535 ? gy : 65535));
        pack_x_kernel<<<grid, block, 0, stream>>>(fields, nv, N1, N2, n2, n3, g2, g3, out);
    } else {
        int64_t na, nj, nq, gq, sa, sq, da, dq;
        if (dir == 1) {
            na = N2; nj = n1; nq = n3; gq = g3;
            sa = N1; sq = N1 * N2; da = N2; dq = N2 * n1;
        } else {
            na = N3; nj = n1; nq = n2; gq = g2;
            sa = N1 * N2; sq = N1; da = N3 * n2; dq = N3;
        }
        const int64_t tiles_a = (na + kTile - 1) / kTile, tiles_j = (nj + kTile - 1) / kTile;
        const int64_t blocks = tiles_a * tiles_j * nq;
        if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
        const int64_t plane = na * nj * nq;
        pack_transpose_kernel<<<(unsigned)blocks, dim3(kTile, kRows), 0, stream>>>(
            fields, nv, na, nj, nq, g1, gq, sa, sq, da, dq, plane, tiles_a, tiles_j, out);
    }
    ++*launches;
    return cudaGetLastError();
}

}  // namespace fvf
