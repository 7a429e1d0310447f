// diffuse2d.cu -- explicit 2D 5-point diffusion step (FP32 and FP64) with
// ping-pong buffers, for sm_103a.
//
// Operation (Qiita, "Fortran 2018 GPU acceleration, part 3", section 3 and
// section 5.1): for interior cells
//     dst(i,j) = c + alpha*((((W + E) + S) + N) - 4c)
// and dst = 0 on the four edges, with the field column-major (i contiguous,
// section 4).  Every operation is rounded to nearest even on its own, in the
// order written: the round-to-nearest intrinsics below are never contracted
// into fused multiply-adds.  In FP64 the single fused operation used,
// fma(-4, c, s), rounds the exact value s - 4c once, which is what s - fl(4c)
// gives whenever 4c is representable (4c is a power-of-two scaling, exact
// unless it overflows); cells with |c| >= 2^1022 take the two-operation form
// instead, so the result is bit-identical for every input.  (The fused form
// saves one FP64 operation; FP32 uses the two operations as written.)
//
// Kernels
//   march  (rows 16-byte aligned, nx a multiple of the vector width): one
//          thread owns one 16-byte vector of cells (4 FP32 or 2 FP64) of a
//          column strip and walks down the strip, keeping the rows j-1, j,
//          j+1 in registers and prefetching row j+2, so every element is
//          read from HBM once per step (plus one row per strip boundary).
//          The W/E neighbours across vectors come from the adjacent lanes by
//          warp shuffle; the two warp-edge lanes load their outside
//          neighbour together with the row.  FP32: the grid is one wave, as
//          many blocks as fit on the SMs at once, each taking an equal band
//          of rows; FP64: bands of 24 rows of 64-thread blocks (many waves,
//          see kMarchF64Rows).
//   scalar (any size or alignment): one thread per cell.
//   blocked (FP32, nsteps >= 3): up to 8 steps per launch in shared memory.
//   cluster (grids of up to 32K cells, nsteps >= 2): all steps in one
//          launch, the grid in the shared memory of a 16-block (8 where the
//          device or the grid does not allow 16) thread-block cluster.
// FP64 takes the cluster kernel or one march (or scalar) launch per step.
// The cluster, blocked and march kernels are described below.
#include <atomic>

#include <cooperative_groups.h>

// The FP64 update reads bit patterns word by word (fp64_emu.cuh): 6% faster
// per 8192^2 step on GB300 than the 64-bit reinterpretation.
#define FVF_EMU_BITS_HILO 1
#include "fp64_emu.cuh"
#include "fvf_internal.cuh"

namespace cg = cooperative_groups;

namespace fvf {
namespace {

template <typename T>
struct Rn;

// s - fl(4c) with two roundings, for the cells where 4c overflows.  Kept out
// of line so that the compiler does not evaluate it for every cell.
static __device__ __noinline__ double sub4_two_ops(double s, double c) {
    return __dsub_rn(s, __dmul_rn(4.0, c));
}

template <>
struct Rn<double> {
    static __device__ __forceinline__ double add(double a, double b) { return __dadd_rn(a, b); }
    static __device__ __forceinline__ double mul(double a, double b) { return __dmul_rn(a, b); }
    // s - 4c rounded once.
    static __device__ __forceinline__ double sub4(double s, double c) {
        if ((__double2hiint(c) & 0x7ff00000) >= 0x7fd00000)  // |c| >= 2^1022, NaN, Inf
            return sub4_two_ops(s, c);
        return __fma_rn(-4.0, c, s);
    }
};

template <>
struct Rn<float> {
    static __device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
    // FP32 arithmetic is cheap: the two rounded operations as written, no
    // fused form and no range check.
    static __device__ __forceinline__ float sub4(float s, float c) {
        return __fsub_rn(s, __fmul_rn(4.0f, c));
    }
};

// Every operation on the arithmetic unit of its precision.
template <typename T>
__device__ __forceinline__ T update_hw(T c, T w, T e, T s, T n, T alpha) {
    using R = Rn<T>;
    const T sum = R::add(R::add(R::add(w, e), s), n);
    return R::add(c, R::mul(alpha, R::sub4(sum, c)));
}

template <typename T>
__device__ __forceinline__ T update(T c, T w, T e, T s, T n, T alpha) {
    return update_hw<T>(c, w, e, s, n, alpha);
}

// FP64 update with the first two neighbour sums (W + E, then + S) on the
// integer pipes (fp64_emu.cuh) and the rest on the FP64 unit: the same
// operations in the same order, each correctly rounded, so the same bits.
// This split balances the two kinds of pipe on GB300 (8192^2 step with the
// march kernel: 0.557 ms, against 0.652 ms with all three sums emulated one
// by one, 0.664 ms with one, 0.787 ms with none; moving alpha * t or the last
// addition too measured slower).  The march kernel now takes the frame form
// below for its same-sign rows; this one serves the kernels whose lanes may
// diverge around the update (scalar, cluster).
template <>
__device__ __forceinline__ double update<double>(double c, double w, double e, double s,
                                                 double n, double alpha) {
    double sum = emu::add_same_sign(w, e);
    sum = emu::add_same_sign(sum, s);
    sum = __dadd_rn(sum, n);
    return __dadd_rn(c, __dmul_rn(alpha, Rn<double>::sub4(sum, c)));
}

// The same update with the whole neighbour sum ((W + E) + S) + N taken in
// one 64-bit fixed-point frame on the integer pipes
// (emu::sum4_one_sign_fast: one alignment and one packing for the three
// additions, each still rounded as binary64 rounds it, the operands
// accumulated with integer multiply-adds) and s - 4c, alpha * t and c + ...
// on the FP64 unit.  The caller guarantees that W, E, S and N have one sign.
// Lanes whose operands the frame declines (a spread of more than 9 binades,
// zeros, subnormals, values at or above 2^1021) take the three additions on
// the FP64 unit in an out-of-line function on bit patterns: a call is not
// if-converted, so lanes that succeed issue no FP64 instruction for the sum
// (written inline, the compiler evaluated the fallback's three additions for
// every cell, 0.78 ms per 8192^2 step).  Measured on GB300 per 8192^2 step,
// with the 12-row bands of the march grid: 0.413 ms, against 0.524 ms with
// update<double> on the same grid.
static __device__ __noinline__ uint64_t sum4_fp64_unit(uint64_t w, uint64_t e, uint64_t s,
                                                       uint64_t n) {
    return emu::bits(__dadd_rn(__dadd_rn(__dadd_rn(emu::from_bits(w), emu::from_bits(e)),
                                         emu::from_bits(s)),
                               emu::from_bits(n)));
}

// ZSLOT (0 = W, 1 = E, -1 = none): the neighbour that may be a zero the
// frame still takes, the face-side neighbour of a cell next to an x edge
// (with two cells per lane: W for the odd cell, E for the even one).  `face`
// marks a cell whose result is discarded (an edge cell): it never calls the
// fallback.  Together they keep the two warps of a row that hold an x edge
// off the fallback on fields with zero edges.
template <typename T, int ZSLOT>
struct Frame {
    static __device__ __forceinline__ T update(T c, T w, T e, T s, T n, T alpha, bool face) {
        (void)face;
        return ::fvf::update<T>(c, w, e, s, n, alpha);
    }
};

template <int ZSLOT>
struct Frame<double, ZSLOT> {
    static __device__ __forceinline__ double update(double c, double w, double e, double s,
                                                    double n, double alpha, bool face) {
        uint64_t sum;
        if (!emu::sum4_one_sign_fast<ZSLOT>(emu::bits(w), emu::bits(e), emu::bits(s),
                                            emu::bits(n), &sum) &&
            !face)
            sum = sum4_fp64_unit(emu::bits(w), emu::bits(e), emu::bits(s), emu::bits(n));
        return __dadd_rn(c, __dmul_rn(alpha, Rn<double>::sub4(emu::from_bits(sum), c)));
    }
};

// The same update for rows where some lane's operands differ in sign.  The
// same-sign form above sends a pair of opposite signs to the complete
// integer algorithm (inline, long), which made a field of mixed signs
// (N(0,1)) 1.84x slower per 8192^2 step on GB300 (1.00 against 0.545 ms).
// Here each addition takes the general integer fast path (either sign), and
// the lanes it declines (ties with shifted-out bits, cancellation, zeros,
// non-normal values) take the FP64 unit, decided by a warp vote so that a
// warp whose lanes all succeed issues no FP64 instruction for it: 0.578 ms
// per step on the N(0,1) field.  Every lane of the warp must call it (the
// march kernel computes it for every cell of such a row, edges included,
// and selects afterwards).
__device__ __forceinline__ double add_any_sign(double a, double b) {
    uint64_t r;
    const bool ok = emu::add_fast_int(emu::bits(a), emu::bits(b), &r);
    if (__all_sync(0xffffffffu, ok)) return emu::from_bits(r);
    return ok ? emu::from_bits(r) : __dadd_rn(a, b);
}

template <typename T>
__device__ __forceinline__ T update_any_sign(T c, T w, T e, T s, T n, T alpha) {
    return update<T>(c, w, e, s, n, alpha);
}

template <>
__device__ __forceinline__ double update_any_sign<double>(double c, double w, double e, double s,
                                                          double n, double alpha) {
    double sum = add_any_sign(w, e);
    sum = add_any_sign(sum, s);
    sum = __dadd_rn(sum, n);
    return __dadd_rn(c, __dmul_rn(alpha, Rn<double>::sub4(sum, c)));
}

// Whether the four neighbours have one sign, the precondition of the
// fixed-point sum (FP64; FP32 has no integer-pipe additions).
template <typename T>
__device__ __forceinline__ bool same_sign4(T w, T e, T s, T n) {
    if constexpr (sizeof(T) == 8) {
        const int hw = __double2hiint(w);
        return ((hw ^ __double2hiint(e)) | (hw ^ __double2hiint(s)) | (hw ^ __double2hiint(n))) >= 0;
    } else {
        return true;
    }
}

// ---------------------------------------------------------------------------
// Scalar kernel (any size, any element alignment)
// ---------------------------------------------------------------------------

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
        if (!FVF_IN(c, nx * ny)) continue;
        if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1) {
            dst[c] = T(0);
        } else if (FVF_IN(c - nx, nx * ny) && FVF_IN(c + nx, nx * ny)) {
            dst[c] = update<T>(src[c], src[c - 1], src[c + 1], src[c - nx], src[c + nx], alpha);
        }
    }
}

// ---------------------------------------------------------------------------
// Row-marching vector kernel
// ---------------------------------------------------------------------------

template <typename T>
struct Vec16;
template <>
struct Vec16<float> {
    static constexpr int n = 4;
    float v[4];
};
template <>
struct Vec16<double> {
    static constexpr int n = 2;
    double v[2];
};

template <typename T>
__device__ __forceinline__ Vec16<T> load16(const T *p) {
    Vec16<T> r;
    if constexpr (sizeof(T) == 4) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p));
        r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
    } else {
        const double2 q = __ldg(reinterpret_cast<const double2 *>(p));
        r.v[0] = q.x; r.v[1] = q.y;
    }
    return r;
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const Vec16<T> &r) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(r.v[0], r.v[1], r.v[2], r.v[3]);
    } else {
        *reinterpret_cast<double2 *>(p) = make_double2(r.v[0], r.v[1]);
    }
}

// Threads per block: FP32 128; FP64 64 (per 8192^2 FP64 step on GB300,
// with bands of 24 rows: 0.4018 ms, against 0.4037 with 128 threads and
// 12 rows, 0.4076 with 256 or with 32 threads).
template <typename T>
__host__ __device__ constexpr int march_threads() { return sizeof(T) == 8 ? 64 : 128; }

// One row of a thread's strip: the vector plus the two scalar neighbours
// that lanes 0 and 31 fetch for the warp (unused in other lanes).
template <typename T>
struct MarchRow {
    Vec16<T> c;
    T w_out, e_out;
};

template <typename T>
__device__ __forceinline__ MarchRow<T> march_load(const T *__restrict__ src, int64_t nx,
                                                  int64_t ny, int64_t j, int64_t col, int lane,
                                                  bool active) {
    constexpr int V = Vec16<T>::n;
    MarchRow<T> r;
#pragma unroll
    for (int k = 0; k < V; ++k) r.c.v[k] = T(0);
    r.w_out = T(0);
    r.e_out = T(0);
    if (active && j >= 0 && j < ny && FVF_IN(nx * j + col + V - 1, nx * ny)) {
        const T *row = src + nx * j;
        r.c = load16<T>(row + col);
        if (lane == 0 && col > 0) r.w_out = __ldg(row + col - 1);
        if (lane == 31 && col + V < nx) r.e_out = __ldg(row + col + V);
    }
    return r;
}

// FP64 rows per block.  The FP64 grid is many short bands rather than one
// wave of long ones: warps whose lanes often take the FP64 fallback (the
// columns next to the zero edges, every row) run slower than the rest, and
// with one wave of long bands the SMs idled while those finished (warps
// active 51% of the SM's capacity against 75% possible).  Short bands let
// the block scheduler even the load out; the extra halo rows (2 per band)
// come from L2 and the kernel is not bound by HBM.  Per 8192^2 step on
// GB300: one wave 0.498 ms; bands of 32, 16, 12, 8 and 6 rows 0.424, 0.414,
// 0.413, 0.415 and 0.419 ms (no register cap; a 40-register cap for 12
// blocks per SM measured 0.416 ms at 12 rows).  With the zero slots and the
// edge cells kept off the fallback (march_rows), bands of 12 and 24 rows
// measure within 0.2% of each other and one wave is still 14% slower; with
// 64-thread blocks 24 rows measured 0.4018 ms against 0.4034 for 12.
constexpr int kMarchF64Rows = 24;
// The rows of one band.  ZX: the block holds an x edge, and its frame sums
// take the zero slots (the other blocks skip the zero tests, whose integer
// instructions measured more than the edge warps' fallback calls cost: on
// every block, 0.424 against 0.414 ms per 8192^2 step; on the edge blocks
// only, 0.404).
template <typename T, bool ZX>
__device__ __forceinline__ void march_rows(const T *__restrict__ src, T *__restrict__ dst,
                                           int64_t nx, int64_t ny, int64_t rows_per_block,
                                           T alpha) {
    constexpr int V = Vec16<T>::n;
    const int lane = threadIdx.x & 31;
    const int64_t col = ((int64_t)blockIdx.x * march_threads<T>() + threadIdx.x) * V;
    const bool active = col < nx;
    const int64_t j0 = (int64_t)blockIdx.y * rows_per_block;
    const int64_t j1 = min(j0 + rows_per_block, ny);

    MarchRow<T> rs = march_load<T>(src, nx, ny, j0 - 1, col, lane, active);
    MarchRow<T> rc = march_load<T>(src, nx, ny, j0, col, lane, active);
    MarchRow<T> rn = march_load<T>(src, nx, ny, j0 + 1, col, lane, active);
    for (int64_t j = j0; j < j1; ++j) {
        const MarchRow<T> rnn = march_load<T>(src, nx, ny, j + 2, col, lane, active);
        // W neighbour of element 0 and E neighbour of element V-1.
        T w_in = __shfl_up_sync(0xffffffffu, rc.c.v[V - 1], 1);
        T e_in = __shfl_down_sync(0xffffffffu, rc.c.v[0], 1);
        if (lane == 0) w_in = rc.w_out;
        if (lane == 31) e_in = rc.e_out;
        Vec16<T> out;
        const bool edge_row = (j == 0) || (j == ny - 1);
        // FP64: one vote per row picks the fixed-point neighbour sum when
        // W, E, S and N have one sign in every lane (every lane takes part:
        // the loop over rows is uniform in the block)
        bool same = true;
#pragma unroll
        for (int k = 0; k < V; ++k)
            same &= same_sign4<T>(k > 0 ? rc.c.v[k - 1] : w_in, k < V - 1 ? rc.c.v[k + 1] : e_in,
                                  rs.c.v[k], rn.c.v[k]);
        if (sizeof(T) == 4 || __all_sync(0xffffffffu, same)) {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const T w = k > 0 ? rc.c.v[k - 1] : w_in;
                const T e = k < V - 1 ? rc.c.v[k + 1] : e_in;
                const int64_t i = col + k;
                const bool edge = edge_row || i == 0 || i == nx - 1;
                // k is a constant in each unrolled copy
                const T val =
                    ZX && V == 2 && k == 0
                        ? Frame<T, 1>::update(rc.c.v[k], w, e, rs.c.v[k], rn.c.v[k], alpha, edge)
                    : ZX && V == 2
                        ? Frame<T, 0>::update(rc.c.v[k], w, e, rs.c.v[k], rn.c.v[k], alpha, edge)
                        : Frame<T, -1>::update(rc.c.v[k], w, e, rs.c.v[k], rn.c.v[k], alpha, edge);
                out.v[k] = edge ? T(0) : val;
            }
        } else {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const T w = k > 0 ? rc.c.v[k - 1] : w_in;
                const T e = k < V - 1 ? rc.c.v[k + 1] : e_in;
                const int64_t i = col + k;
                const bool edge = edge_row || i == 0 || i == nx - 1;
                // computed in every lane (its additions vote), then selected
                const T val = update_any_sign<T>(rc.c.v[k], w, e, rs.c.v[k], rn.c.v[k], alpha);
                out.v[k] = edge ? T(0) : val;
            }
        }
        if (active && FVF_IN(nx * j + col + V - 1, nx * ny)) store16<T>(dst + nx * j + col, out);
        rs = rc;
        rc = rn;
        rn = rnn;
    }
}

template <typename T>
__global__ void __launch_bounds__(march_threads<T>())
diffuse_march_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t nx, int64_t ny,
                     int64_t rows_per_block, T alpha) {
    // block-uniform: the first and last column blocks hold the x edges
    if (sizeof(T) == 8 && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1))
        march_rows<T, true>(src, dst, nx, ny, rows_per_block, alpha);
    else
        march_rows<T, false>(src, dst, nx, ny, rows_per_block, alpha);
}

template <typename T>
int march_blocks_per_sm() {
    // per device; concurrent first calls compute and store the same value
    static std::atomic<int> cached[64];
    const int d = device_slot();
    int n = cached[d].load(std::memory_order_relaxed);
    if (n == 0) {
        const cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, diffuse_march_kernel<T>, march_threads<T>(), 0);
        if (st != cudaSuccess) cudaGetLastError();   // this query's own error only
        if (st != cudaSuccess || n <= 0) n = 8;
        cached[d].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ---------------------------------------------------------------------------
// Temporally blocked kernel: up to kTbSteps steps per launch in shared memory
// ---------------------------------------------------------------------------
//
// A block owns a kTbX x kTbY tile of the output and stages the tile plus a
// halo of kTbSteps cells on every side (a kTbW x kTbH region) in shared
// memory.  Step s (1-based) is valid on the rows and columns at distance >= s
// from the region's border; after `steps` steps the tile is valid and is
// written out.  Every cell receives exactly the update() of the global
// stepping, same operands, same order, so the result is bit-identical; the
// halo is recomputed by the neighbouring tiles.
//
// Work mapping: warp w owns the band of kTbRows rows starting at w*kTbRows
// across the whole region width, each lane four consecutive columns.  A lane
// walks down its band with the rows above and at the current cell in
// registers: per row it loads the row below as one 16-byte shared access (two
// for FP64), takes the W/E neighbours inside its four columns from registers
// and the two outside ones from the adjacent lanes by shuffle, and stores the
// four results with one access.  Rows outside the valid range of a step are
// skipped (the bound is uniform in the warp); all columns are computed: a
// column outside the valid range computes values that are never read by a
// valid cell (influence travels one cell per step).  Global edge cells are
// set to zero at every step; cells outside the grid are never read by an
// interior cell.
constexpr int kTbSteps = 8;
constexpr int kTbX = 112, kTbY = 64;
constexpr int kTbW = kTbX + 2 * kTbSteps;   // 128 = 4 columns per lane
constexpr int kTbH = kTbY + 2 * kTbSteps;   // 80
constexpr int kTbThreads = 256;             // 8 warps
constexpr int kTbRows = kTbH / 8;           // rows per warp band
constexpr int kTbCx = kTbW / 32;
static_assert(kTbW == 128 && kTbH % 8 == 0, "tile shape: one warp spans a row, 4 columns per lane");

// Four consecutive elements of a shared-memory row (16-byte aligned).
template <typename T>
struct Quad {
    T v[4];
};

template <typename T>
__device__ __forceinline__ Quad<T> ld_quad(const T *p) {
    Quad<T> q;
    if constexpr (sizeof(T) == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(p);
        q.v[0] = x.x; q.v[1] = x.y; q.v[2] = x.z; q.v[3] = x.w;
    } else {
        const double2 x = reinterpret_cast<const double2 *>(p)[0];
        const double2 y = reinterpret_cast<const double2 *>(p)[1];
        q.v[0] = x.x; q.v[1] = x.y; q.v[2] = y.x; q.v[3] = y.y;
    }
    return q;
}

template <typename T>
__device__ __forceinline__ void st_quad(T *p, const Quad<T> &q) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(q.v[0], q.v[1], q.v[2], q.v[3]);
    } else {
        reinterpret_cast<double2 *>(p)[0] = make_double2(q.v[0], q.v[1]);
        reinterpret_cast<double2 *>(p)[1] = make_double2(q.v[2], q.v[3]);
    }
}

// Two blocks per SM is what the shared memory allows in FP32 (80 KB each).
template <typename T>
__global__ void __launch_bounds__(kTbThreads, 2)
diffuse_tblock_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t nx, int64_t ny,
                      int steps, T alpha) {
    extern __shared__ unsigned char smem_raw[];
    T *buf0 = reinterpret_cast<T *>(smem_raw);
    T *buf1 = buf0 + kTbW * kTbH;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gi0 = (int64_t)blockIdx.x * kTbX - kTbSteps;
    const int64_t gj0 = (int64_t)blockIdx.y * kTbY - kTbSteps;

    // stage the region (rows strided over the warps: coalesced 32-wide rows)
#pragma unroll
    for (int b = 0; b < kTbH / 8; ++b) {
        const int lj = warp + 8 * b;
        const int64_t gj = gj0 + lj;
#pragma unroll
        for (int a = 0; a < kTbCx; ++a) {
            const int li = lane + 32 * a;
            const int64_t gi = gi0 + li;
            T val = T(0);
            if (gi >= 0 && gi < nx && gj >= 0 && gj < ny && FVF_IN(gi + nx * gj, nx * ny))
                val = __ldg(src + gi + nx * gj);
            buf0[lj * kTbW + li] = val;
        }
    }
    // The second buffer starts as zeros: the columns computed outside the
    // valid range then stay finite (left-over shared memory could hold bit
    // patterns that send every such cell down the rare-value path).
    for (int idx = threadIdx.x; idx < kTbW * kTbH / 4; idx += kTbThreads) {
        Quad<T> z;
#pragma unroll
        for (int k = 0; k < 4; ++k) z.v[k] = T(0);
        st_quad<T>(buf1 + 4 * idx, z);
    }
    const int li0 = 4 * lane;                    // this lane's four columns
    bool col_edge[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t gi = gi0 + li0 + k;
        col_edge[k] = gi == 0 || gi == nx - 1;
    }
    __syncthreads();

    const int band0 = warp * kTbRows;
    for (int s = 1; s <= steps; ++s) {
        const T *in = (s & 1) ? buf0 : buf1;
        T *out = (s & 1) ? buf1 : buf0;
        const int r0 = max(band0, s), r1 = min(band0 + kTbRows, kTbH - s);
        if (r0 < r1) {          // uniform in the warp
            Quad<T> up = ld_quad<T>(in + (r0 - 1) * kTbW + li0);
            Quad<T> cur = ld_quad<T>(in + r0 * kTbW + li0);
            const int gjb = (int)gj0;            // row r is global row gjb + r
            // one row: results into out, returns the row below
            auto row = [&](int r, const Quad<T> &above, const Quad<T> &mid) -> Quad<T> {
                const Quad<T> below = ld_quad<T>(in + (r + 1) * kTbW + li0);
                const T w_in = __shfl_up_sync(0xffffffffu, mid.v[3], 1);
                const T e_in = __shfl_down_sync(0xffffffffu, mid.v[0], 1);
                const int gj = gjb + r;
                const bool row_edge = gj == 0 || gj == (int)ny - 1;
                Quad<T> res;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const T w = k > 0 ? mid.v[k - 1] : w_in;
                    const T e = k < 3 ? mid.v[k + 1] : e_in;
                    const T val = update<T>(mid.v[k], w, e, above.v[k], below.v[k], alpha);
                    res.v[k] = (row_edge || col_edge[k]) ? T(0) : val;
                }
                st_quad<T>(out + r * kTbW + li0, res);
                return below;
            };
            int r = r0;
            for (; r + 1 < r1; r += 2) {          // two rows per trip: no copies
                const Quad<T> b1 = row(r, up, cur);
                const Quad<T> b2 = row(r + 1, cur, b1);
                up = b1;
                cur = b2;
            }
            if (r < r1) row(r, up, cur);
        }
        __syncthreads();
    }

    const T *fin = (steps & 1) ? buf1 : buf0;
#pragma unroll
    for (int b = 0; b < kTbH / 8; ++b) {
        const int lj = warp + 8 * b;
        const int64_t gj = gj0 + lj;
        if (lj < kTbSteps || lj >= kTbSteps + kTbY || gj < 0 || gj >= ny) continue;
#pragma unroll
        for (int a = 0; a < kTbCx; ++a) {
            const int li = lane + 32 * a;
            const int64_t gi = gi0 + li;
            if (li >= kTbSteps && li < kTbSteps + kTbX && gi >= 0 && gi < nx &&
                FVF_IN(gi + nx * gj, nx * ny))
                dst[gi + nx * gj] = fin[lj * kTbW + li];
        }
    }
}

// ---------------------------------------------------------------------------
// Cluster kernel: a small grid in the shared memory of one thread-block
// cluster, every step in one launch
// ---------------------------------------------------------------------------
//
// For grids of up to a few tens of thousands of cells the time goes to
// launch latency and, for FP64, to arithmetic that one SM would do alone.  A
// cluster of 8 or 16 blocks (one per SM) splits the rows into bands:
// each block keeps both ping-pong states of its band in its own shared
// memory, reads the row just above and just below its band from the
// neighbouring blocks' shared memory (distributed shared memory), and the
// blocks separate steps with the cluster barrier (a hardware barrier: every
// block of a cluster is resident at once).  Each cell gets the same update()
// as in the other kernels, so the same bits.  At the end every block writes
// its band of the last state to the result array and of the state before it
// to the other array.
constexpr int kClusterThreads = 512;
constexpr int64_t kClusterMaxBytes = 200 * 1024;   // per block: both states of a band
// Largest grid the cluster kernel takes.  Measured on GB300 (16-block
// cluster against the per-step march kernel for FP64 and the blocked kernel
// for FP32): 128^2 x 100 steps 237 vs 425 us (FP64) and 89 vs 151 us (FP32);
// 200^2 x 50 steps 243 vs 220 us and 85 vs 87 us; larger grids favour the
// others.
constexpr int64_t kClusterMaxCells = 32 * 1024;

// CS blocks per cluster, launched with the cluster dimension as a launch
// attribute.  A thread's cells (c = tid, tid + blockDim.x, ...) are the same
// at every step; their (row, column) are stepped by a fixed increment rather
// than divided out per cell and step.  HW: the FP64 update entirely on the
// FP64 unit, for bands of at most kClusterHwCells cells, where a step is
// bound by the latency of one cell's update rather than by throughput (the
// integer-pipe additions lengthen that chain).  In one A/B on GB300 (the
// same box, call by call): 64^2 x 32 steps 43 us with this form against
// 48 us with the split, and 128^2 x 100 steps 246 against 238 us (the split
// wins there).
constexpr int kClusterHwCells = 512;

template <typename T, int CS, bool HW>
__global__ void __launch_bounds__(kClusterThreads)
diffuse_cluster_kernel(const T *__restrict__ u0, T *__restrict__ u, T *__restrict__ v, int nx,
                       int ny, int band, int64_t nsteps, T alpha) {
    extern __shared__ unsigned char smem_raw[];
    T *const st0 = reinterpret_cast<T *>(smem_raw);
    T *const st1 = st0 + band * nx;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int r0 = rank * band;
    const int rows = max(0, min(band, ny - r0));
    const int cells = rows * nx;
    const int nt = (int)blockDim.x;
    const int step_r = nt / nx, step_i = nt - step_r * nx;
    const int lr0 = (int)threadIdx.x / nx, i0 = (int)threadIdx.x - lr0 * nx;
    for (int c = threadIdx.x; c < cells; c += nt)
        if (FVF_IN((int64_t)r0 * nx + c, (int64_t)nx * ny)) st0[c] = u0[(int64_t)r0 * nx + c];
    cluster.sync();
    for (int64_t s = 1; s <= nsteps; ++s) {
        T *in = (s & 1) ? st0 : st1;
        T *out = (s & 1) ? st1 : st0;
        // the neighbours' copies of the same state (rows r0-1 and r0+rows)
        const T *above = rank > 0 ? cluster.map_shared_rank(in, rank - 1) : nullptr;
        const T *below = rank + 1 < CS ? cluster.map_shared_rank(in, rank + 1) : nullptr;
        int lr = lr0, i = i0;
        for (int c = threadIdx.x; c < cells; c += nt) {
            const int j = r0 + lr;
            if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1) {
                out[c] = T(0);
            } else {
                const T sv = lr > 0 ? in[c - nx] : above[(band - 1) * nx + i];
                const T nv = lr + 1 < rows ? in[c + nx] : below[i];
                out[c] = HW ? update_hw<T>(in[c], in[c - 1], in[c + 1], sv, nv, alpha)
                            : update<T>(in[c], in[c - 1], in[c + 1], sv, nv, alpha);
            }
            lr += step_r;
            i += step_i;
            if (i >= nx) {
                i -= nx;
                ++lr;
            }
        }
        cluster.sync();
    }
    // state n is in st[n & 1]; it belongs in v for odd n and in u for even n
    const T *last = (nsteps & 1) ? st1 : st0, *prev = (nsteps & 1) ? st0 : st1;
    T *res = (nsteps & 1) ? v : u, *oth = (nsteps & 1) ? u : v;
    for (int c = threadIdx.x; c < cells; c += nt) {
        if (!FVF_IN((int64_t)r0 * nx + c, (int64_t)nx * ny)) continue;
        res[(int64_t)r0 * nx + c] = last[c];
        oth[(int64_t)r0 * nx + c] = prev[c];
    }
}

// Band height for a cluster of cs blocks, 0 when the cluster kernel does not
// apply (nsteps >= 2: step n-1 must exist for the other buffer).
template <typename T>
int cluster_band(int64_t nx, int64_t ny, int64_t nsteps, int cs) {
    if (nsteps < 2 || nx > 65536 || ny > 65536 || nx * ny > kClusterMaxCells) return 0;
    const int64_t band = (ny + cs - 1) / cs;
    if (band * nx * 2 * (int64_t)sizeof(T) > kClusterMaxBytes) return 0;
    return (int)band;
}

// Per device, once: the dynamic shared-memory attribute of both kernels, and
// whether a 16-block (non-portable) cluster of the largest band can be
// resident.  Returns the widest usable cluster: 16, 8, or 0 for none.
template <typename T>
int cluster_prepare() {
    static std::atomic<int> width1[64];   // width + 1 once known (0: not yet)
    const int d = device_slot();
    const int known = width1[d].load(std::memory_order_relaxed);
    if (known) return known - 1;
    // An attribute or occupancy query that fails leaves its error as the
    // thread's last error; it is cleared here (so that the launch checks that
    // follow do not report it) only when one of these calls failed.
    bool failed = false;
    auto ok = [&failed](cudaError_t e) {
        if (e != cudaSuccess) failed = true;
        return e == cudaSuccess;
    };
    int w = 0;
    if (ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 8, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kClusterMaxBytes)) &&
        ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 8, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kClusterMaxBytes)))
        w = 8;
    if (w &&
        ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 16, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kClusterMaxBytes)) &&
        ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 16, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kClusterMaxBytes)) &&
        ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 16, false>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) &&
        ok(cudaFuncSetAttribute(diffuse_cluster_kernel<T, 16, true>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1))) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kClusterThreads);
        cfg.dynamicSmemBytes = (size_t)kClusterMaxBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // both instantiations a 16-block launch may take (all-FP64 update for
        // bands of up to kClusterHwCells cells, the split one above that)
        int c0 = 0, c1 = 0;
        if (ok(cudaOccupancyMaxActiveClusters(&c0, diffuse_cluster_kernel<T, 16, false>, &cfg)) &&
            ok(cudaOccupancyMaxActiveClusters(&c1, diffuse_cluster_kernel<T, 16, true>, &cfg)) &&
            c0 > 0 && c1 > 0)
            w = 16;
    }
    if (failed) cudaGetLastError();
    width1[d].store(w + 1, std::memory_order_relaxed);
    return w;
}

template <typename T, int CS>
cudaError_t launch_cluster(T *u, T *v, int nx, int ny, int band, int64_t nsteps, T alpha,
                           cudaStream_t stream) {
    // threads: the band's cells rounded up to a warp, at most kClusterThreads
    const int cells = band * nx;
    const int threads = cells >= kClusterThreads ? kClusterThreads : ((cells + 31) / 32) * 32;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(CS);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = (size_t)(2 * cells) * sizeof(T);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // u is both the input and an output: every block reads its band before
    // the first cluster barrier and writes after the last.
    if (cells <= kClusterHwCells)
        return cudaLaunchKernelEx(&cfg, diffuse_cluster_kernel<T, CS, true>, (const T *)u, u, v,
                                  nx, ny, band, nsteps, alpha);
    return cudaLaunchKernelEx(&cfg, diffuse_cluster_kernel<T, CS, false>, (const T *)u, u, v, nx,
                              ny, band, nsteps, alpha);
}

constexpr size_t tblock_smem_bytes(size_t elem) { return 2 * (size_t)kTbW * kTbH * elem; }

// Whether to run blocks of steps in shared memory (FP32 only): FP32 is
// HBM-bound, so blocking cuts its traffic about sixfold.  FP64 is bound by
// its arithmetic, and a block of steps puts a tile's whole multi-step work on
// one SM: measured 3x slower than a launch per step even at 1024^2 (778 vs
// 258 us for 20 steps) and far slower on grids of fewer tiles than SMs.
template <typename T>
bool use_tblock(int64_t nx, int64_t ny, int64_t nsteps) {
    if (sizeof(T) != 4 || nsteps < 3) return false;
    const int64_t tiles_y = (ny + kTbY - 1) / kTbY;
    return tiles_y <= 65535 && (nx + kTbX - 1) / kTbX <= 0x7fffffff;
}

template <typename T>
cudaError_t tblock_prepare() {
    static std::atomic<int> status1[64];  // status + 1 once known (0: not yet)
    const int d = device_slot();
    const int known = status1[d].load(std::memory_order_relaxed);
    if (known) return (cudaError_t)(known - 1);
    const cudaError_t st = cudaFuncSetAttribute(diffuse_tblock_kernel<T>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)tblock_smem_bytes(sizeof(T)));
    if (st != cudaSuccess) cudaGetLastError();
    status1[d].store((int)st + 1, std::memory_order_relaxed);
    return st;
}

// One-step launches (march or scalar kernel), configured once per call.
template <typename T>
struct SingleStep {
    bool vec_ok = false;
    dim3 grid, block;
    int64_t rows = 0;

    cudaError_t setup(const T *u, const T *v, int64_t nx, int64_t ny) {
        constexpr int V = Vec16<T>::n;
        vec_ok = (nx % V == 0) && ((uintptr_t)u % 16 == 0) && ((uintptr_t)v % 16 == 0) &&
                 nx >= 2 * V;
        if (vec_ok) {
            constexpr int kThreads = march_threads<T>();
            const int64_t bx = (nx / V + kThreads - 1) / kThreads;
            int64_t by;
            if (sizeof(T) == 8) {
                // bands of kMarchF64Rows rows (more where the grid's y
                // dimension would exceed its limit)
                rows = kMarchF64Rows;
                if ((ny + rows - 1) / rows > 65535) rows = (ny + 65534) / 65535;
            } else {
                // FP32: one wave of equal bands
                const int64_t resident = (int64_t)march_blocks_per_sm<T>() * sm_count();
                by = resident / bx;
                if (by < 1) by = 1;
                if (by > ny) by = ny;
                rows = (ny + by - 1) / by;
            }
            by = (ny + rows - 1) / rows;
            if (bx > 0x7fffffff || by > 65535) return cudaErrorInvalidValue;
            grid = dim3((unsigned)bx, (unsigned)by);
            block = dim3(kThreads);
        } else {
            const int64_t gy = (ny + kBy - 1) / kBy;
            grid = dim3((unsigned)((nx + kBx - 1) / kBx), (unsigned)(gy < 65535 ? gy : 65535));
            block = dim3(kBx, kBy);
        }
        return cudaSuccess;
    }

    void launch(const T *src, T *dst, int64_t nx, int64_t ny, T alpha, cudaStream_t stream) {
        if (vec_ok)
            diffuse_march_kernel<T><<<grid, block, 0, stream>>>(src, dst, nx, ny, rows, alpha);
        else
            diffuse_step_kernel<T><<<grid, block, 0, stream>>>(src, dst, nx, ny, alpha);
    }
};

template <typename T>
cudaError_t run(T *u, T *v, int64_t nx, int64_t ny, T alpha, int64_t nsteps,
                cudaStream_t stream, uint64_t *launches) {
    cudaError_t e;
    // small grids (both states of an eighth of the grid fit one block's
    // shared memory): all steps in one cluster launch, of 16 blocks where the
    // device allows a cluster that wide and the grid has two rows per block
    const int width =
        cluster_band<T>(nx, ny, nsteps, 8) ? cluster_prepare<T>() : 0;
    if (width) {
        if (width == 16 && ny >= 32) {
            const int band = cluster_band<T>(nx, ny, nsteps, 16);
            e = launch_cluster<T, 16>(u, v, (int)nx, (int)ny, band, nsteps, alpha, stream);
        } else {
            const int band = cluster_band<T>(nx, ny, nsteps, 8);
            e = launch_cluster<T, 8>(u, v, (int)nx, (int)ny, band, nsteps, alpha, stream);
        }
        if (e != cudaSuccess) return e;
        ++*launches;
        return cudaGetLastError();
    }
    SingleStep<T> one;
    e = one.setup(u, v, nx, ny);
    if (e != cudaSuccess) return e;
    // FP32 only: FP64 takes one launch per step (see use_tblock)
    if constexpr (sizeof(T) == 4) {
        if (use_tblock<T>(nx, ny, nsteps) && tblock_prepare<T>() == cudaSuccess) {
            // Steps 1..n-1 in B blocked launches, step n as one single-step
            // launch, so the other buffer ends holding step n-1.  Launch k reads
            // u (k even) or v (k odd); step n-1 must end in u when n is odd (the
            // last step writes v) and in v when n is even, i.e. B must have the
            // parity of n+1.  B = n-1 (one step per launch) always has it, so
            // raising B by one when needed keeps B <= n-1.
            const int64_t n1 = nsteps - 1;
            int64_t nb = (n1 + kTbSteps - 1) / kTbSteps;
            if ((nb & 1) != ((nsteps + 1) & 1)) ++nb;
            const dim3 grid((unsigned)((nx + kTbX - 1) / kTbX),
                            (unsigned)((ny + kTbY - 1) / kTbY));
            const size_t smem = tblock_smem_bytes(sizeof(T));
            for (int64_t k = 0; k < nb; ++k) {
                const int steps = (int)(n1 / nb + (k < n1 % nb ? 1 : 0));
                const T *src = (k & 1) ? v : u;
                T *dst = (k & 1) ? u : v;
                diffuse_tblock_kernel<T><<<grid, kTbThreads, smem, stream>>>(src, dst, nx, ny,
                                                                              steps, alpha);
                ++*launches;
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
            const T *src = (nsteps & 1) ? u : v;
            T *dst = (nsteps & 1) ? v : u;
            one.launch(src, dst, nx, ny, alpha, stream);
            ++*launches;
            return cudaGetLastError();
        }
    }
    for (int64_t s = 1; s <= nsteps; ++s) {
        const T *src = (s & 1) ? u : v;
        T *dst = (s & 1) ? v : u;
        one.launch(src, dst, nx, ny, alpha, stream);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

FVF_BOUNDS_READER(read_bounds_diffuse2d)

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
