// weno_pack.cu -- multi-variable WENO input pack for sm_103a.
//
// Operation (MFlowCode/MFC pull request #2087, "Changes",
// s_pack_weno_input_arr): out(a,b,c,i) = field_i(...) with the swept axis
// first (x: no permutation; y: j and k exchanged; z: j and l exchanged), the
// swept axis covering its ghost cells and the transverse axes their interior.
// A pure 64-bit copy.  The same file holds the conservative-variable copy
// (s_compute_rhs on the same page) alone and fused with the pack: the pack
// reads the fields the copy reads, so the fused pass reads them once.
//
// Mapping ("Why this is faster" on the same page): one thread per spatial
// output cell, the variable loop sequential inside the thread, the index
// arithmetic done once per cell and reused for every variable.  x keeps the
// contiguous index on the lanes for both the load and the store.  y and z are
// transposes: a block of 128 threads stages a 32 x 32 tile of each variable
// in shared memory so that both the global load (along j) and the global
// store (along the swept axis) are coalesced.
#include "fvf_internal.cuh"

namespace fvf {
namespace {

constexpr int kTile = 32;
// Threads along the second tile axis of the transposing kernel (each thread
// then moves kTile / rows elements of a variable's tile).  4 rows (8 elements
// per thread, 128-thread blocks) measured 3-5% faster on GB300 than 8 rows,
// and 16 rows 12-25% slower; 2 rows equal in FP32, slower in FP64.
constexpr int kPackRows = 4;
// Minimum resident blocks per SM of the transposing kernel: FP32 at 12 (a
// 40-register cap, 12 blocks of 128 threads) keeps enough 4-byte loads in
// flight per SM for HBM (8 x 207^3, y: 0.113 -> 0.107 ms, z: 0.123 -> 0.115 ms
// on GB300); FP64 moves twice the bytes per thread and measured slower with
// the cap (spills), so it takes none.
template <typename T>
constexpr int pack_min_blocks() { return sizeof(T) == 4 ? 12 : 0; }

// x: out(a, b, c, i) = f_i(a, b+g2, c+g3); (M1, M2, M3) = (N1, n2, n3).
// For a fixed c the n2 rows of N1 elements are one contiguous run in the
// source (a spans the whole stored axis, b the interior rows) and in the
// packed output, so the kernel copies each run of N1*n2 elements with a
// flat index: blockIdx.y walks c, blockIdx.x a chunk of the run, and no lane
// idles on rows whose length is not a multiple of the block width (a 64-wide
// block over 207-element rows left 19% of the lanes idle).  K elements per
// thread and variable: 4 in FP32 (8 x 207^3 on GB300: 0.089 -> 0.084 ms),
// 1 in FP64 (HBM-bound either way, 0.159 ms).  T is double or float: the
// pack is a copy of 8- or 4-byte elements.
constexpr int kPackXThreads = 256;
template <typename T>
__host__ __device__ constexpr int pack_x_per_thread() { return sizeof(T) == 4 ? 4 : 1; }

template <typename T>
__global__ void __launch_bounds__(kPackXThreads)
pack_x_kernel(FieldTable t, int nv, int64_t N1, int64_t N2, int64_t n2, int64_t n3,
              int64_t g2, int64_t g3, T *__restrict__ out) {
    constexpr int K = pack_x_per_thread<T>();
    const int64_t len = N1 * n2;                 // one c plane of the output
    const int64_t plane = len * n3;              // one variable of the output
    const int64_t stored = N1 * N2 * (n3 + 2 * g3);
    (void)stored;
    const int64_t e0 = (int64_t)blockIdx.x * (kPackXThreads * K) + threadIdx.x;
    bool ok[K];
#pragma unroll
    for (int k = 0; k < K; ++k) ok[k] = e0 + k * kPackXThreads < len;
    for (int64_t c = blockIdx.y; c < n3; c += gridDim.y) {
        const int64_t src = N1 * (g2 + N2 * (c + g3)) + e0;
        const int64_t dst = c * len + e0;
        for (int i = 0; i < nv; ++i) {
            const T *f = static_cast<const T *>(t.p[i]) + src;
            T v[K];
#pragma unroll
            for (int k = 0; k < K; ++k)
                v[k] = ok[k] && FVF_IN(src + k * kPackXThreads, stored)
                           ? __ldg(f + k * kPackXThreads) : T(0);
            T *o = out + (int64_t)i * plane + dst;
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (ok[k] && FVF_IN(dst + k * kPackXThreads + (int64_t)i * plane, plane * nv))
                    o[k * kPackXThreads] = v[k];
        }
    }
}

// Transposing pack (y or z), optionally fused with the conservative-variable
// copy.  The tile spans the swept axis (output-fast, index a, 0..na-1) and the
// j axis (input-fast, index jt, 0..nj-1); the third axis (index q, 0..nq-1)
// is fixed per block.
//   source element    (jt + jo) + sa*a + sq*(q + qo)
//   packed element    a + da*(jt - pj) + dq*(q - pq), written when
//                     0 <= jt - pj < pnj and 0 <= q - pq < pnq
// Pack alone: jt and q run over the interior (jo, qo = the ghost offsets,
// pj = pq = 0).  Pack with copy: jt and q run over the whole stored box
// (jo = qo = 0, pj, pq = the ghost offsets) and every loaded element is also
// stored to its copy at the source index, a coalesced store along j.
//   y: a = k, jt = j, q = l; packed extents (N2, n1, n3)
//   z: a = l, jt = j, q = k; packed extents (N3, n2, n1)
// The tile is double-buffered across variables: the loads of variable i+1
// are in flight while variable i is stored, with one barrier per variable.

struct TransposeGeom {
    int64_t na, nj, nq, jo, qo, pj, pq, pnj, pnq, sa, sq, da, dq, plane, tiles_a, tiles_j;
    int64_t stored;  // elements of one field's stored box (index checks)
};

template <typename T, bool COPY, typename Idx, int R>
__global__ void __launch_bounds__(kTile * R, pack_min_blocks<T>())
pack_transpose_kernel(FieldTable t, CopyTable cp, int nv, TransposeGeom G,
                      T *__restrict__ out) {
    // geometry in the index type of this instantiation: 32-bit when every
    // index the block forms fits (the launcher checks), else 64-bit
    const Idx na = (Idx)G.na, nj = (Idx)G.nj, jo = (Idx)G.jo, qo = (Idx)G.qo;
    const Idx pj = (Idx)G.pj, pq = (Idx)G.pq, pnj = (Idx)G.pnj, pnq = (Idx)G.pnq;
    const Idx sa = (Idx)G.sa, sq = (Idx)G.sq, da = (Idx)G.da, dq = (Idx)G.dq;
    const Idx plane = (Idx)G.plane, tiles_a = (Idx)G.tiles_a, tiles_j = (Idx)G.tiles_j;
    const Idx stored = (Idx)G.stored;
    constexpr int TA = kTile;            // tile extent along a
    constexpr int LP = kTile / R;        // loads per thread and variable
    constexpr int kRows = R, kPer = LP;
    __shared__ T tile[2][TA][kTile + 1];
    Idx blk = (Idx)blockIdx.x;
    const Idx ta = blk % tiles_a;
    blk /= tiles_a;
    const Idx tj = blk % tiles_j;
    const Idx q = blk / tiles_j;
    const Idx a0 = ta * TA, j0 = tj * kTile;
    const int tx = threadIdx.x, ty = threadIdx.y;
    // load side: lanes along j (contiguous in the field), rows along a
    const Idx jl = j0 + tx;
    const Idx src0 = (jl + jo) + sa * (a0 + ty) + sq * (q + qo);
    bool lok[LP];
#pragma unroll
    for (int r = 0; r < LP; ++r) lok[r] = jl < nj && a0 + ty + r * kRows < na;
    const Idx qp = q - pq;
    if (COPY && (qp < 0 || qp >= pnq)) {
        // a transverse ghost slice: copied, not packed (block-uniform branch)
        for (int i = 0; i < nv; ++i) {
            const T *f = static_cast<const T *>(t.p[i]);
            T *c = reinterpret_cast<T *>(cp.p[i]);
            T v[LP];
#pragma unroll
            for (int r = 0; r < LP; ++r)
                v[r] = lok[r] && FVF_IN(src0 + sa * (r * kRows), stored)
                           ? __ldg(f + src0 + sa * (r * kRows)) : T(0);
#pragma unroll
            for (int r = 0; r < LP; ++r)
                if (lok[r] && FVF_IN(src0 + sa * (r * kRows), stored))
                    c[src0 + sa * (r * kRows)] = v[r];
        }
        return;
    }
    // store side: lanes along a (contiguous in the output), rows along j
    const Idx jp0 = j0 + ty - pj;
    const Idx dst0 = a0 + tx + da * jp0 + dq * qp;
    bool sok[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const Idx jp = jp0 + r * kRows;
        sok[r] = a0 + tx < na && jp >= 0 && jp < pnj;
    }

    T v[LP];
    {
        const T *f = static_cast<const T *>(t.p[0]);
#pragma unroll
        for (int r = 0; r < LP; ++r)
            v[r] = lok[r] && FVF_IN(src0 + sa * (r * kRows), stored)
                       ? __ldg(f + src0 + sa * (r * kRows)) : T(0);
#pragma unroll
        for (int r = 0; r < LP; ++r) tile[0][ty + r * kRows][tx] = v[r];
        if (COPY) {
            T *c = reinterpret_cast<T *>(cp.p[0]);
#pragma unroll
            for (int r = 0; r < LP; ++r)
                if (lok[r] && FVF_IN(src0 + sa * (r * kRows), stored))
                    c[src0 + sa * (r * kRows)] = v[r];
        }
    }
    __syncthreads();
    for (int i = 0; i < nv; ++i) {
        const int buf = i & 1;
        const bool more = i + 1 < nv;
        if (more) {
            const T *f = static_cast<const T *>(t.p[i + 1]);
#pragma unroll
            for (int r = 0; r < LP; ++r)
                v[r] = lok[r] && FVF_IN(src0 + sa * (r * kRows), stored)
                           ? __ldg(f + src0 + sa * (r * kRows)) : T(0);
        }
        const Idx obase = (Idx)i * plane + dst0;
#pragma unroll
        for (int r = 0; r < kPer; ++r)
            if (sok[r] && FVF_IN(obase + da * (r * kRows), plane * nv))
                out[obase + da * (r * kRows)] = tile[buf][tx][ty + r * kRows];
        if (more) {
#pragma unroll
            for (int r = 0; r < LP; ++r) tile[buf ^ 1][ty + r * kRows][tx] = v[r];
            if (COPY) {
                T *c = reinterpret_cast<T *>(cp.p[i + 1]);
#pragma unroll
                for (int r = 0; r < LP; ++r)
                    if (lok[r] && FVF_IN(src0 + sa * (r * kRows), stored))
                        c[src0 + sa * (r * kRows)] = v[r];
            }
        }
        __syncthreads();
    }
}

// x pack fused with the copy, with the flat index of the x pack: blockIdx.y
// walks the stored planes c, blockIdx.x a chunk of the plane's N1*N2
// contiguous elements.  Each element is loaded once and stored to its copy,
// and to the packed output when it lies in a transverse-interior row (a
// contiguous run of N1*n2 elements of an interior plane).  Variables go in
// batches of kBatch: the batch's loads are issued before its stores, so they
// overlap even though the compiler cannot prove the copies and the fields
// apart.
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kPackXThreads, 4)
pack_copy_x_kernel(FieldTable t, CopyTable cp, int nv, int64_t N1, int64_t N2, int64_t N3,
                   int64_t n2, int64_t n3, int64_t g2, int64_t g3, double *__restrict__ out) {
    const int64_t sp = N1 * N2;                  // one stored plane
    const int64_t len = N1 * n2;                 // its packed rows
    const int64_t plane = len * n3;
    const int64_t e = (int64_t)blockIdx.x * kPackXThreads + threadIdx.x;
    if (e >= sp) return;
    const int64_t pe = e - N1 * g2;              // position in the packed rows
    for (int64_t c = blockIdx.y; c < N3; c += gridDim.y) {
        const int64_t pc = c - g3;
        const bool packed = pe >= 0 && pe < len && pc >= 0 && pc < n3;
        const int64_t src = c * sp + e;
        const int64_t dst = pc * len + pe;
        const bool sin = FVF_IN(src, sp * N3);
        for (int i0 = 0; i0 < nv; i0 += kBatch) {
            double x[kBatch];
#pragma unroll
            for (int r = 0; r < kBatch; ++r)
                if (i0 + r < nv && sin)
                    x[r] = __ldg(static_cast<const double *>(t.p[i0 + r]) + src);
#pragma unroll
            for (int r = 0; r < kBatch; ++r) {
                if (i0 + r < nv && sin) {
                    cp.p[i0 + r][src] = x[r];
                    if (packed && FVF_IN((int64_t)(i0 + r) * plane + dst, plane * nv))
                        out[(int64_t)(i0 + r) * plane + dst] = x[r];
                }
            }
        }
    }
}

// The copy alone over the flat stored box: one thread per element (per pair
// of elements with 16-byte vectors when every pointer allows it), variables in
// batches as above, grid-stride over one wave of blocks.
template <bool V2>
__global__ void __launch_bounds__(256)
fields_copy_kernel(FieldTable t, CopyTable cp, int nv, int64_t total) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (V2) {
        const int64_t pairs = total >> 1;
        for (int64_t e = tid; e < pairs; e += stride) {
            if (!FVF_IN(2 * e + 1, total)) continue;
            for (int i0 = 0; i0 < nv; i0 += kBatch) {
                double2 x[kBatch];
#pragma unroll
                for (int r = 0; r < kBatch; ++r)
                    if (i0 + r < nv)
                        x[r] = __ldg(reinterpret_cast<const double2 *>(t.p[i0 + r]) + e);
#pragma unroll
                for (int r = 0; r < kBatch; ++r)
                    if (i0 + r < nv) reinterpret_cast<double2 *>(cp.p[i0 + r])[e] = x[r];
            }
        }
        if ((total & 1) && tid == 0)
            for (int i = 0; i < nv; ++i)
                cp.p[i][total - 1] = __ldg(static_cast<const double *>(t.p[i]) + total - 1);
    } else {
        for (int64_t e = tid; e < total; e += stride) {
            for (int i0 = 0; i0 < nv; i0 += kBatch) {
                double x[kBatch];
#pragma unroll
                for (int r = 0; r < kBatch; ++r)
                    if (i0 + r < nv) x[r] = __ldg(static_cast<const double *>(t.p[i0 + r]) + e);
#pragma unroll
                for (int r = 0; r < kBatch; ++r)
                    if (i0 + r < nv) cp.p[i0 + r][e] = x[r];
            }
        }
    }
}

}  // namespace

FVF_BOUNDS_READER(read_bounds_pack)

// Launch geometry of the transposing kernel for dir 1 or 2 (see above).
static TransposeGeom transpose_geom(const Box &box, int dir, bool copy) {
    const int64_t n1 = box.n[0], n2 = box.n[1], n3 = box.n[2];
    const int64_t N1 = box.N[0], N2 = box.N[1], N3 = box.N[2];
    const int64_t g1 = box.g[0];
    TransposeGeom G;
    int64_t nq, Nq, gq;
    if (dir == 1) {
        G.na = N2; nq = n3; Nq = N3; gq = box.g[2];
        G.sa = N1; G.sq = N1 * N2; G.da = N2; G.dq = N2 * n1;
        G.plane = N2 * n1 * n3;
    } else {
        G.na = N3; nq = n2; Nq = N2; gq = box.g[1];
        G.sa = N1 * N2; G.sq = N1; G.da = N3 * n2; G.dq = N3;
        G.plane = N3 * n2 * n1;
    }
    G.pnj = n1;
    G.pnq = nq;
    G.stored = N1 * N2 * N3;
    if (copy) {
        G.nj = N1; G.nq = Nq; G.jo = 0; G.qo = 0; G.pj = g1; G.pq = gq;
    } else {
        G.nj = n1; G.nq = nq; G.jo = g1; G.qo = gq; G.pj = 0; G.pq = 0;
    }
    G.tiles_a = (G.na + kTile - 1) / kTile;
    G.tiles_j = (G.nj + kTile - 1) / kTile;
    return G;
}

template <typename T, bool COPY>
static cudaError_t launch_transpose(const FieldTable &fields, const CopyTable &copies, int nv,
                                    const Box &box, int dir, T *out, cudaStream_t stream) {
    const TransposeGeom G = transpose_geom(box, dir, COPY);
    const int64_t blocks = G.tiles_a * G.tiles_j * G.nq;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    // 32-bit indices (fewer registers, more blocks per SM: 4-8% faster at
    // 8 x 207^3) while every index a block forms, including those of the rows
    // and columns past the box edge that it computes but does not use, fits
    const int64_t lim = (int64_t)1 << 31;
    const bool narrow = G.stored + 32 * G.sa + G.sq + 64 < lim &&
                        G.plane * nv + 40 * G.da + G.dq + 64 < lim && blocks < lim;
    constexpr int R = kPackRows;
    if (narrow)
        pack_transpose_kernel<T, COPY, int32_t, R><<<(unsigned)blocks, dim3(kTile, R), 0,
                                                     stream>>>(fields, copies, nv, G, out);
    else
        pack_transpose_kernel<T, COPY, int64_t, R><<<(unsigned)blocks, dim3(kTile, R), 0,
                                                     stream>>>(fields, copies, nv, G, out);
    return cudaSuccess;
}

template <typename T>
static cudaError_t launch_pack_typed(const FieldTable &fields, int nv, const Box &box, int dir,
                                     T *out, cudaStream_t stream) {
    const int64_t n2 = box.n[1], n3 = box.n[2];
    const int64_t N1 = box.N[0], N2 = box.N[1];
    const int64_t g2 = box.g[1], g3 = box.g[2];
    if (dir == 0) {
        const int64_t chunk = (int64_t)kPackXThreads * pack_x_per_thread<T>();
        const int64_t gx = (N1 * n2 + chunk - 1) / chunk;
        if (gx > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)gx, (unsigned)(n3 < 65535 ? n3 : 65535));
        pack_x_kernel<T><<<grid, kPackXThreads, 0, stream>>>(fields, nv, N1, N2, n2, n3, g2, g3,
                                                            out);
        return cudaSuccess;
    }
    CopyTable none;
    for (int i = 0; i < kMaxNv; ++i) none.p[i] = nullptr;
    return launch_transpose<T, false>(fields, none, nv, box, dir, out, stream);
}

cudaError_t launch_weno_pack(const FieldTable &fields, int nv, const Box &box, int dir,
                             void *out, bool fp32, cudaStream_t stream, uint64_t *launches) {
    const cudaError_t e =
        fp32 ? launch_pack_typed<float>(fields, nv, box, dir, static_cast<float *>(out), stream)
             : launch_pack_typed<double>(fields, nv, box, dir, static_cast<double *>(out), stream);
    if (e != cudaSuccess) return e;
    ++*launches;
    return cudaGetLastError();
}

cudaError_t launch_weno_pack_copy(const FieldTable &fields, int nv, const Box &box, int dir,
                                  double *out, const CopyTable &copies, cudaStream_t stream,
                                  uint64_t *launches) {
    if (dir == 0) {
        const int64_t N1 = box.N[0], N2 = box.N[1], N3 = box.N[2];
        const int64_t gx = (N1 * N2 + kPackXThreads - 1) / kPackXThreads;
        if (gx > 0x7fffffff) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)gx, (unsigned)(N3 < 65535 ? N3 : 65535));
        pack_copy_x_kernel<<<grid, kPackXThreads, 0, stream>>>(fields, copies, nv, N1, N2, N3,
                                                              box.n[1], box.n[2], box.g[1],
                                                              box.g[2], out);
    } else {
        const cudaError_t e =
            launch_transpose<double, true>(fields, copies, nv, box, dir, out, stream);
        if (e != cudaSuccess) return e;
    }
    ++*launches;
    return cudaGetLastError();
}

cudaError_t launch_fields_copy(const FieldTable &fields, int nv, int64_t stored,
                               const CopyTable &copies, cudaStream_t stream, uint64_t *launches) {
    bool v2 = true;
    for (int i = 0; i < nv; ++i)
        v2 = v2 && ((uintptr_t)fields.p[i] % 16 == 0) && ((uintptr_t)copies.p[i] % 16 == 0);
    const int64_t work = v2 ? (stored >> 1) + 1 : stored;
    int64_t blocks = (work + 255) / 256;
    const int64_t wave = (int64_t)sm_count() * 8;
    if (blocks > wave) blocks = wave;
    if (v2)
        fields_copy_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(fields, copies, nv, stored);
    else
        fields_copy_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(fields, copies, nv, stored);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace fvf
