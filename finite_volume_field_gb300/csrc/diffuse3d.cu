// diffuse3d.cu -- explicit 3D 7-point diffusion step (FP32 and FP64) with
// ping-pong buffers, for sm_103a.
//
// Operation: the 3D variant of the update of Qiita, "Fortran 2018 GPU
// acceleration, part 3" (section 3, with the edges of section 5.1 and the
// ping-pong of section 5.4): for interior cells
//     dst(i,j,k) = c + alpha*((((((W + E) + S) + N) + B) + T) - 6c)
// with W/E the i-1/i+1, S/N the j-1/j+1 and B/T the k-1/k+1 neighbours, and
// dst = 0 on the six boundary faces.  Column-major layout, i contiguous:
// cell (i,j,k) at i + nx*(j + ny*k).  Every operation is rounded to nearest
// even on its own in the order written; 6c is its own rounded product (6c is
// not a power-of-two scaling, so no fused form is exact here).
//
// Kernels (both march along k; a block owns a tile of 32*V cells along i
// by a few rows along j, V = 4 FP32 or 2 FP64 cells per lane).
//   bulk   (FP32, rows 16-byte aligned: nx a multiple of 4, 16-byte
//          buffers): 4 warps, a tile of 8 rows (each warp computes two).
//          One thread streams whole planes of the tile into a ring of
//          shared-memory slots with tensor-map bulk copies
//          (cp.async.bulk.tensor), two planes ahead of the plane being
//          computed.  A plane is one (32V+2V) x 10 box: the tile's
//          rows plus one halo row above and below, each widened by 16 bytes
//          on both sides for the W/E neighbours; the copy engine zero-fills
//          the parts outside the grid, and one mbarrier per slot counts the
//          bytes in.  Every cell then reads c, W, E, S, N, B and T from the
//          staged planes k-1, k and k+1, so HBM sees each element once per
//          step (the halo rows and the planes at the ends of a run are the
//          only re-reads, mostly from L2).  The grid is persistent: about as
//          many blocks as fit at once, each taking an equal number of (tile,
//          run of planes) items.  Every mbarrier wait is bounded; if one
//          expires the block records it in a device flag (fvf_device_error),
//          waits (bounded) for its copies in flight and returns.
//   march  (FP64, and FP32 rows that are not 16-byte aligned; V cells per
//          lane, 1 when unaligned): each lane keeps planes k-1, k, k+1 of its
//          cells in registers and prefetches k+2; W/E by warp shuffle, S/N
//          from the tile's rows staged in shared memory.  FP64: runs of 16
//          planes (many waves of blocks); FP32: the planes split into runs so
//          that about 8 blocks per SM are in flight.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "fp64_emu.cuh"
#include "fvf_internal.cuh"
#include "mbarrier.cuh"

// How the FP64 update splits its work between the FP64 unit and the integer
// pipes (fp64_emu.cuh): the five neighbour sums (W+E, +S, +N, +B, +T, in that
// order) run in one fixed-point frame on the integer pipes where the six
// operands have one sign and span at most 8 binades (emu::sum_one_sign_fast;
// a zero W or E, the face-side neighbour of a cell next to an x face, is
// taken too); 6c, the subtraction, alpha * (...) and the last addition run on
// the FP64 unit (4 instructions per cell).  Per 512^3 step on GB300: 1.56 ms
// before the zero slots (1.48 ms with them, in a build that measured the
// former at 1.70), against 1.85 ms with two sums and both products on the
// integer pipes (1.68 ms with the frame and both products there: the ALU
// pipe saturates).  Every split gives the same bits.  Aligned FP32 grids take the bulk-copy kernel; FP64
// takes the register march kernel, which measured faster there (FP64
// arithmetic, not memory, bounds the FP64 update).

namespace fvf {
namespace {

constexpr int kTY = 4;  // warps per block of the bulk kernel

__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }

__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }

template <typename T>
__device__ __forceinline__ T update3(T c, T w, T e, T s, T n, T b, T t, T alpha) {
    T x = add_rn(w, e);
    x = add_rn(x, s);
    x = add_rn(x, n);
    x = add_rn(x, b);
    x = add_rn(x, t);
    return add_rn(c, mul_rn(alpha, sub_rn(x, mul_rn(T(6), c))));
}

// FP32 update of two cells at once for the bulk kernel: the additions as
// packed two-lane FP32 instructions (add.rn.f32x2, each lane an IEEE
// round-to-nearest addition), the products 6c and alpha * (...) as scalar
// multiplications.  A packed product whose only use is a packed addition is
// contracted into one packed fused multiply-add by the compiler, even with
// explicit .rn and --fmad=false (measured on GB300: the fused result in 100%
// of cases); scalar products feeding a packed addition are not.  11
// instructions for two cells instead of 18: 0.212 -> 0.197 ms per 512^3
// step, bit-identical.  (In the 2D blocked kernel the same form measured
// slower: building the lane pairs costs more there.)
__device__ __forceinline__ unsigned long long pack2(float x, float y) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 unpack2(unsigned long long r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ unsigned long long add2_rn(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float2 update3x2(float2 c, float2 w, float2 e, float2 s, float2 n,
                                           float2 b, float2 t, float alpha) {
    unsigned long long x = add2_rn(pack2(w.x, w.y), pack2(e.x, e.y));
    x = add2_rn(x, pack2(s.x, s.y));
    x = add2_rn(x, pack2(n.x, n.y));
    x = add2_rn(x, pack2(b.x, b.y));
    x = add2_rn(x, pack2(t.x, t.y));
    // x - 6c as x + (-6c): the same rounded result
    const float2 d = unpack2(add2_rn(x, pack2(__fmul_rn(-6.0f, c.x), __fmul_rn(-6.0f, c.y))));
    return unpack2(add2_rn(pack2(c.x, c.y), pack2(__fmul_rn(alpha, d.x), __fmul_rn(alpha, d.y))));
}

// The five neighbour sums on the FP64 unit, for the lanes whose operands the
// fixed-point frame declines (zeros such as the boundary neighbours, signs
// that differ, spreads over 8 binades, subnormals, values from 2^1021 up).
// Out of line on bit patterns: a call is not if-converted, so lanes that
// take the frame issue no FP64 instruction for the sum.
static __device__ __noinline__ uint64_t sum6_fp64_unit(uint64_t w, uint64_t e, uint64_t s,
                                                       uint64_t n, uint64_t b, uint64_t t) {
    double x = __dadd_rn(emu::from_bits(w), emu::from_bits(e));
    x = __dadd_rn(x, emu::from_bits(s));
    x = __dadd_rn(x, emu::from_bits(n));
    x = __dadd_rn(x, emu::from_bits(b));
    return emu::bits(__dadd_rn(x, emu::from_bits(t)));
}

// FP64 update.  ZSLOT (0 = W, 1 = E, -1 = none) is the neighbour that may be
// a zero the frame still takes (the face-side neighbour of the cells next to
// an x face: with two cells per lane that is W for the odd cell and E for the
// even one).  `face` marks a cell whose result is discarded (a boundary
// face cell): it never calls the fallback.  Per 512^3 step on GB300, in one
// build: 1.703 ms with neither, 1.622 with the face cells' calls left out,
// 1.485 with the zero slots too (bit-identical; the two warps of eight in a
// 512-wide row that hold an x face no longer take the fallback).
template <int ZSLOT>
__device__ __forceinline__ double update3_fp64(double c, double w, double e, double s, double n,
                                               double b, double t, double alpha, bool face) {
    const uint64_t X[6] = {emu::bits(w), emu::bits(e), emu::bits(s),
                           emu::bits(n), emu::bits(b), emu::bits(t)};
    uint32_t h[6];
#pragma unroll
    for (int q = 0; q < 6; ++q) h[q] = (uint32_t)(X[q] >> 32);
    // a zero in the slot takes its partner's sign for the test
    if constexpr (ZSLOT >= 0) {
        if (emu::is_zero_bits(X[ZSLOT])) h[ZSLOT] = h[1 - ZSLOT];
    }
    const bool one_sign = (int)((h[0] ^ h[1]) | (h[0] ^ h[2]) | (h[0] ^ h[3]) |
                                (h[0] ^ h[4]) | (h[0] ^ h[5])) >= 0;
    uint64_t sum;
    const bool ok = emu::sum_one_sign_fast<6, ZSLOT>(X, &sum);
    if (!(ok && one_sign) && !face) sum = sum6_fp64_unit(X[0], X[1], X[2], X[3], X[4], X[5]);
    return __dadd_rn(c, __dmul_rn(alpha, __dsub_rn(emu::from_bits(sum), __dmul_rn(6.0, c))));
}

template <typename T, int V>
struct Vec {
    T v[V];
};

// Loads this lane's vector of row `row` (cells x0 + lane*V .. +V-1; zeros
// past the end) and, for lanes 0 and 31, the outside neighbour of the warp's
// segment (x0 - 1 and x0 + 32V; zero where it does not exist).
// `off` is the row's offset in its nx*ny*nz array (index checks only).
template <typename T, int V>
__device__ __forceinline__ void load_row(const T *__restrict__ row, int64_t x0, int lane,
                                         int64_t nx, Vec<T, V> &out, T &xh, int64_t off,
                                         int64_t total) {
    (void)off; (void)total;
    const int64_t xi = x0 + (int64_t)lane * V;
    if (xi < nx && FVF_IN(off + xi + V - 1, total)) {
        if constexpr (V == 4) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(row + xi));
            out.v[0] = q.x; out.v[1] = q.y; out.v[2] = q.z; out.v[3] = q.w;
        } else if constexpr (V == 2) {
            const double2 q = __ldg(reinterpret_cast<const double2 *>(row + xi));
            out.v[0] = q.x; out.v[1] = q.y;
        } else {
            out.v[0] = __ldg(row + xi);
        }
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) out.v[v] = T(0);
    }
    const int64_t xo = lane == 0 ? x0 - 1 : x0 + 32 * V;
    xh = ((lane == 0 || lane == 31) && xo >= 0 && xo < nx && FVF_IN(off + xo, total))
             ? __ldg(row + xo) : T(0);
}

template <typename T, int V>
__device__ __forceinline__ void store_row(T *__restrict__ row, int64_t x0, int lane, int64_t nx,
                                          const Vec<T, V> &x, int64_t off, int64_t total) {
    (void)off; (void)total;
    const int64_t xi = x0 + (int64_t)lane * V;
    if (xi >= nx || !FVF_IN(off + xi + V - 1, total)) return;
    if constexpr (V == 4) {
        *reinterpret_cast<float4 *>(row + xi) = make_float4(x.v[0], x.v[1], x.v[2], x.v[3]);
    } else if constexpr (V == 2) {
        *reinterpret_cast<double2 *>(row + xi) = make_double2(x.v[0], x.v[1]);
    } else {
        row[xi] = x.v[0];
    }
}

template <typename T, int V>
__device__ __forceinline__ void store_vec(T *p, const Vec<T, V> &x) {
    if constexpr (V == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(x.v[0], x.v[1], x.v[2], x.v[3]);
    } else if constexpr (V == 2) {
        *reinterpret_cast<double2 *>(p) = make_double2(x.v[0], x.v[1]);
    } else {
        *p = x.v[0];
    }
}

// Rows (warps) per block of the register march kernel.  FP64: 4.  Per
// 512^3 FP64 step on GB300, runs of 16 planes, 64 registers (8 blocks per
// SM): 1.405 ms with 4 rows, against 1.422 with 2, 1.484 with 6, 1.492 with
// 8 and 1.740 with 16 (1024 threads per SM in each).  With 4 rows and no
// minimum-blocks bound the compiler takes 72 registers (7 blocks per SM):
// 1.354 ms, against 1.377 with a minimum of 6 blocks (also 72 registers),
// 1.406 with 8 (64), 1.409 with 5 (82) and 1.451 with 9 (56, spills).
// FP32 (rows that are not 16-byte aligned): 8.
template <typename T>
__host__ __device__ constexpr int march3_rows() { return sizeof(T) == 8 ? 4 : 8; }

// Every block takes the zero slots: taking them only in the blocks that
// hold an x face (a block-uniform branch between two copies of the loop)
// measured slower, 1.529 against 1.483 ms per step with 8-row tiles (spills
// at the 64-register cap) and 1.402 against 1.353 with 4-row tiles and no
// cap.
template <typename T, int V>
__global__ void __launch_bounds__(32 * march3_rows<T>())
diffuse3d_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t nx, int64_t ny,
                 int64_t nz, T alpha, int64_t kz_len) {
    constexpr int kR = march3_rows<T>();
    __shared__ T rows[2][kR + 2][32 * V];
    const int lane = threadIdx.x, w = threadIdx.y;
    const int64_t x0 = (int64_t)blockIdx.x * (32 * V);
    const int64_t j0 = (int64_t)blockIdx.y * kR;
    const int64_t j = j0 + w;
    const int64_t kz0 = (int64_t)blockIdx.z * kz_len;
    const int64_t kz1 = kz0 + kz_len < nz ? kz0 + kz_len : nz;
    const int64_t sxy = nx * ny;
    const bool rowok = j < ny;
    // halo rows of the tile: warp 0 also carries row j0-1, warp kR-1 row j0+kR
    const int64_t jh = w == 0 ? j0 - 1 : j0 + kR;
    const bool hok = (w == 0 || w == kR - 1) && jh >= 0 && jh < ny;
    const int hslot = w == 0 ? 0 : kR + 1;
    const int64_t klast = kz1 < nz ? kz1 : nz - 1;  // last plane this block reads

    Vec<T, V> prev, cur, next, nn, hcur, hnext, hnn;
    T xp = T(0), xc = T(0), xn = T(0), xnn = T(0), hx;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        prev.v[v] = cur.v[v] = next.v[v] = nn.v[v] = T(0);
        hcur.v[v] = hnext.v[v] = hnn.v[v] = T(0);
    }
    const int64_t total = sxy * nz;
    auto load = [&](int64_t jr, int64_t kp, Vec<T, V> &o, T &h) {
        load_row<T, V>(src + jr * nx + kp * sxy, x0, lane, nx, o, h, jr * nx + kp * sxy, total);
    };
    if (rowok) {
        if (kz0 >= 1) load(j, kz0 - 1, prev, xp);
        load(j, kz0, cur, xc);
        if (kz0 + 1 <= klast) load(j, kz0 + 1, next, xn);
    }
    if (hok) {
        load(jh, kz0, hcur, hx);
        if (kz0 + 1 <= klast) load(jh, kz0 + 1, hnext, hx);
    }
    (void)xp;
    int buf = 0;
    for (int64_t k = kz0; k < kz1; ++k) {
        // stage plane k of the tile's rows (and halo rows) for the S/N reads
        if (rowok) {
#pragma unroll
            for (int v = 0; v < V; ++v) rows[buf][w + 1][lane * V + v] = cur.v[v];
        }
        if (hok) {
#pragma unroll
            for (int v = 0; v < V; ++v) rows[buf][hslot][lane * V + v] = hcur.v[v];
        }
        // prefetch plane k+2
        if (k + 2 <= klast) {
            if (rowok) load(j, k + 2, nn, xnn);
            if (hok) load(jh, k + 2, hnn, hx);
        }
        __syncthreads();
        if (rowok) {
            Vec<T, V> out;
            const bool edge = k == 0 || k == nz - 1 || j == 0 || j == ny - 1;
            // W of the first element and E of the last, from the neighbouring
            // lanes (the warp-edge lanes use their outside neighbour)
            const T wl = __shfl_up_sync(0xffffffffu, cur.v[V - 1], 1);
            const T er = __shfl_down_sync(0xffffffffu, cur.v[0], 1);
            const T wfirst = lane == 0 ? xc : wl;
            const T elast = lane == 31 ? xc : er;
            if (edge) {
#pragma unroll
                for (int v = 0; v < V; ++v) out.v[v] = T(0);
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t i = x0 + (int64_t)lane * V + v;
                    const T we = v == 0 ? wfirst : cur.v[v - 1];
                    const T ea = v == V - 1 ? elast : cur.v[v + 1];
                    const T so = rows[buf][w][lane * V + v];
                    const T no = rows[buf][w + 2][lane * V + v];
                    const bool face = i == 0 || i >= nx - 1;
                    T val;
                    if constexpr (sizeof(T) == 8) {
                        // v is a constant in each unrolled copy
                        if (V == 2 && v == 0)
                            val = update3_fp64<1>(cur.v[v], we, ea, so, no, prev.v[v], next.v[v],
                                                  alpha, face);
                        else if (V == 2)
                            val = update3_fp64<0>(cur.v[v], we, ea, so, no, prev.v[v], next.v[v],
                                                  alpha, face);
                        else
                            val = update3_fp64<-1>(cur.v[v], we, ea, so, no, prev.v[v],
                                                   next.v[v], alpha, face);
                    } else {
                        val = update3<T>(cur.v[v], we, ea, so, no, prev.v[v], next.v[v], alpha);
                    }
                    out.v[v] = face ? T(0) : val;
                }
            }
            store_row<T, V>(dst + j * nx + k * sxy, x0, lane, nx, out, j * nx + k * sxy, total);
        }
        prev = cur;
        cur = next;
        next = nn;
        xc = xn;
        xn = xnn;
        hcur = hnext;
        hnext = hnn;
        buf ^= 1;
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy kernel
// ---------------------------------------------------------------------------

// Blocks of 4 warps, a ring of 5 slots, 2 rows per warp and runs of 128
// planes measured best at 512^3 on GB300 (one box, back to back, 0.169 ms
// per step: 72 registers and 27.7 KB of shared memory, 7 blocks per SM;
// runs of 64, 32 and 16 planes 0.170, 0.174 and 0.179 ms: every run re-reads
// two halo planes).
// Against it: 8 warps 0.197; 4 warps with a ring of 4 or 6 slots 0.191 or
// 0.206 (6 slots fit only 6 blocks); with a 64-register cap for 8 blocks
// 0.182 (spills); with 3 or 4 rows per warp 0.182 or 0.199; 2 warps of 4
// rows 0.189.  (Before the packed additions, 8 warps: 0.216 against 0.240
// for 6 slots, 1 row, 32 planes.)
constexpr int kRing = 5;                     // slots: planes k-1, k, k+1 and kRing-3 ahead
constexpr int kRPW = 2;                      // rows per warp in the bulk kernel
constexpr int64_t kRunPlanes = 128;          // planes per work item of the bulk kernel
constexpr int kBulkRows = kTY * kRPW;        // tile rows of a bulk block
constexpr int kRows = kBulkRows + 2;         // tile rows plus one halo row each side

__device__ int g_device_error;   // bit 1: a bounded wait expired; bit 2: a drain wait too

using mbar::smem_addr;

template <typename T, int V>
__device__ __forceinline__ Vec<T, V> ld_stage(const T *p) {
    Vec<T, V> r;
    if constexpr (V == 4) {
        const float4 q = *reinterpret_cast<const float4 *>(p);
        r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
    } else {
        const double2 q = *reinterpret_cast<const double2 *>(p);
        r.v[0] = q.x; r.v[1] = q.y;
    }
    return r;
}

// Staged row: 32V cells plus a 16-byte margin each side (544 bytes); a slot
// holds kRows of them, padded to the 128-byte alignment of a tensor copy.
template <typename T>
__host__ __device__ constexpr int row_elems() {
    return 32 * (16 / (int)sizeof(T)) + 2 * (16 / (int)sizeof(T));
}
template <typename T>
__host__ __device__ constexpr size_t slot_bytes() {
    return ((size_t)kRows * row_elems<T>() * sizeof(T) + 127) / 128 * 128;
}
template <typename T>
__host__ __device__ constexpr size_t bulk_smem_bytes() {
    return kRing * slot_bytes<T>() + kRing * sizeof(uint64_t) + 128;
}

template <typename T>
__global__ void __launch_bounds__(32 * kTY)
diffuse3d_bulk_kernel(const __grid_constant__ CUtensorMap src_map, T *__restrict__ dst,
                      int64_t nx, int64_t ny, int64_t nz, T alpha, int64_t kz_len,
                      int64_t tiles_x, int64_t tiles_y, int64_t items) {
    constexpr int V = 16 / sizeof(T);        // cells per lane
    constexpr int P = V;                     // 16 bytes of W/E margin each side of a row
    constexpr int TX = 32 * V;
    constexpr int RW = TX + 2 * P;           // staged row length (544 bytes)
    constexpr int64_t SLOT = (int64_t)(slot_bytes<T>() / sizeof(T));  // elements per slot
    constexpr uint32_t kBoxBytes = (uint32_t)(kRows * RW * sizeof(T));
    extern __shared__ unsigned char smem_raw[];
    // 128-byte aligned base for the tensor copies
    unsigned char *base = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    T *stage = reinterpret_cast<T *>(base);  // [kRing][SLOT], rows of RW
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kRing * slot_bytes<T>());
    const int lane = threadIdx.x, w = threadIdx.y;
    const bool producer = lane == 0 && w == 0;
    const int64_t sxy = nx * ny;
    if (producer) {
        for (int s = 0; s < kRing; ++s) mbar::init(smem_addr(&bars[s]), 1);
        mbar::fence_init();
    }
    __syncthreads();
    // Planes are loaded in order and numbered t = 0, 1, ... over all items of
    // this block; plane t sits in slot t % kRing, and its completion is phase
    // number t / kRing of that slot's mbarrier (parity (t / kRing) & 1).
    uint32_t tbase = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t tx = item % tiles_x, rest = item / tiles_x;
        const int64_t ty = rest % tiles_y, run = rest / tiles_y;
        const int64_t x0 = tx * TX, j0 = ty * kBulkRows, kz0 = run * kz_len;
        const int64_t kz1 = kz0 + kz_len < nz ? kz0 + kz_len : nz;
        const int64_t pl0 = kz0 > 0 ? kz0 - 1 : 0;       // planes read: pl0..pl1
        const int64_t pl1 = kz1 < nz ? kz1 : nz - 1;
        // one box per plane: x from x0-P (16 bytes left of the tile), rows
        // j0-1 .. j0+kTY; parts outside the grid arrive as zeros
        auto issue = [&](int64_t p) {
            const uint32_t sl = (tbase + (uint32_t)(p - pl0)) % kRing;
            const uint32_t bar = smem_addr(&bars[sl]);
            mbar::expect_tx(bar, kBoxBytes);
            mbar::tensor_load_3d(smem_addr(stage + (int64_t)sl * SLOT), &src_map, (int)(x0 - P),
                                 (int)(j0 - 1), (int)p, bar);
        };
        auto wait_t = [&](uint32_t t) {
            return mbar::wait(smem_addr(&bars[t % kRing]), (t / kRing) & 1u);
        };
        int64_t issued = pl0 - 1;                         // producer: last plane issued
        if (producer)
            for (int64_t p = pl0; p <= pl1 && p < pl0 + kRing; ++p) {
                issue(p);
                issued = p;
            }
        const int64_t xi = x0 + (int64_t)lane * V;
        // every cell of this lane is interior along i: no per-cell i test
        const bool lane_inner = xi >= 1 && xi + V <= nx - 1;
        // this warp's rows: j0 + w + kTY*r, r < kRPW
        T *drow = dst + (j0 + w) * nx + kz0 * sxy;
        // slots and parities of planes k-1, k, k+1, advanced every plane
        uint32_t tk = tbase + (uint32_t)(kz0 - pl0);
        uint32_t sc = tk % kRing, pc = (tk / kRing) & 1u;
        uint32_t sb = (tk + kRing - 1) % kRing, pb = ((tk + kRing - 1) / kRing + 1) & 1u;
        uint32_t st = (tk + 1) % kRing, pt = ((tk + 1) / kRing) & 1u;
        for (int64_t k = kz0; k < kz1; ++k) {
            bool ok = true;
            if (k - 1 >= pl0) ok = mbar::wait(smem_addr(&bars[sb]), pb) && ok;
            ok = mbar::wait(smem_addr(&bars[sc]), pc) && ok;
            if (k + 1 <= pl1) ok = mbar::wait(smem_addr(&bars[st]), pt) && ok;
            if (__syncthreads_or(!ok)) {
                // a copy did not land in time: record it, let the copies in
                // flight finish (bounded) and leave.  If a drain wait expires
                // too, bit 2 records that the block may have exited with a
                // copy into its shared memory still pending.  (Not exercised
                // by a test: making a tensor copy fail to land would need a
                // fault of the copy engine.)
                if (producer) {
                    atomicOr(&g_device_error, 1);
                    for (int64_t p = k > pl0 ? k - 1 : pl0; p <= issued; ++p)
                        if (!wait_t(tbase + (uint32_t)(p - pl0))) atomicOr(&g_device_error, 2);
                }
                return;
            }
            // every thread is done with plane k-2 (read in the previous
            // iteration): its slot takes the plane kRing-2 ahead of k
            if (producer && k - 2 >= pl0 && k - 2 + kRing <= pl1) {
                issue(k - 2 + kRing);
                issued = k - 2 + kRing;
            }
#pragma unroll
            for (int r = 0; r < kRPW; ++r) {
                const int64_t j = j0 + w + kTY * r;
                if (j >= ny) break;
                Vec<T, V> out;
                const bool edge = k == 0 || k == nz - 1 || j == 0 || j == ny - 1;
                if (edge) {
#pragma unroll
                    for (int v = 0; v < V; ++v) out.v[v] = T(0);
                } else {
                    const int64_t ro = (int64_t)(w + kTY * r + 1) * RW + P + lane * V;
                    const T *rc = stage + (int64_t)sc * SLOT + ro;
                    const T *rb = stage + (int64_t)sb * SLOT + ro;
                    const T *rt = stage + (int64_t)st * SLOT + ro;
                    const Vec<T, V> c = ld_stage<T, V>(rc);
                    const Vec<T, V> so = ld_stage<T, V>(rc - RW);
                    const Vec<T, V> no = ld_stage<T, V>(rc + RW);
                    const Vec<T, V> bo = ld_stage<T, V>(rb);
                    const Vec<T, V> to = ld_stage<T, V>(rt);
                    const T wl = __shfl_up_sync(0xffffffffu, c.v[V - 1], 1);
                    const T er = __shfl_down_sync(0xffffffffu, c.v[0], 1);
                    const T wfirst = lane == 0 ? rc[-1] : wl;      // margin cell x0-1
                    const T elast = lane == 31 ? rc[V] : er;       // margin cell x0+32V
                    T res[V];
                    if constexpr (sizeof(T) == 4) {
                        // two cells per update3x2: (v, v+1) with W (v-1, v), E (v+1, v+2)
#pragma unroll
                        for (int v = 0; v < V; v += 2) {
                            const T w0 = v == 0 ? wfirst : c.v[(v + V - 1) % V];
                            const T e1 = v + 2 < V ? c.v[(v + 2) % V] : elast;
                            const float2 r2 = update3x2(
                                make_float2(c.v[v], c.v[v + 1]), make_float2(w0, c.v[v]),
                                make_float2(c.v[v + 1], e1), make_float2(so.v[v], so.v[v + 1]),
                                make_float2(no.v[v], no.v[v + 1]), make_float2(bo.v[v], bo.v[v + 1]),
                                make_float2(to.v[v], to.v[v + 1]), alpha);
                            res[v] = r2.x;
                            res[v + 1] = r2.y;
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const T we = v == 0 ? wfirst : c.v[v - 1];
                            const T ea = v == V - 1 ? elast : c.v[v + 1];
                            res[v] = update3<T>(c.v[v], we, ea, so.v[v], no.v[v], bo.v[v],
                                                to.v[v], alpha);
                        }
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int64_t i = xi + v;
                        out.v[v] = (lane_inner || (i != 0 && i < nx - 1)) ? res[v] : T(0);
                    }
                }
                T *drw = drow + kTY * r * nx;
                if (xi < nx && FVF_IN((drw - dst) + xi + V - 1, sxy * nz))
                    store_vec<T, V>(drw + xi, out);
            }
            drow += sxy;
            sb = sc; pb = pc;
            sc = st; pc = pt;
            if (++st == kRing) { st = 0; pt ^= 1u; }
        }
        tbase += (uint32_t)(pl1 - pl0 + 1);
        __syncthreads();  // the next item's first copies reuse slots read above
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of a whole nx*ny*nz field, box (32V+2V) x kRows x 1.  False if
// the driver call is unavailable or refuses the map.
template <typename T>
bool encode_field_map(CUtensorMap *map, const T *base, int64_t nx, int64_t ny, int64_t nz) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || nx >= ((int64_t)1 << 32) || ny >= ((int64_t)1 << 32) || nz >= ((int64_t)1 << 31))
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)nx, (cuuint64_t)ny, (cuuint64_t)nz};
    const cuuint64_t strides[2] = {(cuuint64_t)(nx * (int64_t)sizeof(T)),
                                   (cuuint64_t)(nx * ny * (int64_t)sizeof(T))};
    const cuuint32_t box[3] = {(cuuint32_t)row_elems<T>(), (cuuint32_t)kRows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = fn(map, sizeof(T) == 8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT64
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          3, const_cast<T *>(base), dims, strides, box, estride,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T>
cudaError_t launch_bulk(const CUtensorMap &src_map, T *dst, int64_t nx, int64_t ny, int64_t nz,
                        T alpha, cudaStream_t stream) {
    constexpr int TX = 32 * (16 / sizeof(T));
    constexpr size_t smem = bulk_smem_bytes<T>();
    // per device, the attribute and occupancy; concurrent first calls compute
    // and store the same value
    static std::atomic<int> per_sm_dev[64];
    const int d = device_slot();
    int per_sm = per_sm_dev[d].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(diffuse3d_bulk_kernel<T>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return cudaGetLastError();
        int n = 0;
        const cudaError_t st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, diffuse3d_bulk_kernel<T>, 32 * kTY, smem);
        if (st != cudaSuccess) cudaGetLastError();   // this query's own error only
        if (st != cudaSuccess || n < 1) n = 1;
        per_sm = n;
        per_sm_dev[d].store(n, std::memory_order_relaxed);
    }
    const int64_t tiles_x = (nx + TX - 1) / TX, tiles_y = (ny + kBulkRows - 1) / kBulkRows;
    const int64_t kz_len = kRunPlanes;  // planes per item
    const int64_t runs = (nz + kz_len - 1) / kz_len;
    const int64_t items = tiles_x * tiles_y * runs;
    const int64_t maxgrid = (int64_t)per_sm * sm_count();
    const int64_t waves = (items + maxgrid - 1) / maxgrid;
    const int64_t grid = (items + waves - 1) / waves;  // equal items per block
    diffuse3d_bulk_kernel<T><<<(unsigned)grid, dim3(32, kTY), smem, stream>>>(
        src_map, dst, nx, ny, nz, alpha, kz_len, tiles_x, tiles_y, items);
    return cudaSuccess;
}

template <typename T, int V>
cudaError_t launch_typed(const T *src, T *dst, int64_t nx, int64_t ny, int64_t nz, T alpha,
                         cudaStream_t stream) {
    const int64_t gx = (nx + 32 * V - 1) / (32 * V);
    constexpr int kR = march3_rows<T>();
    const int64_t gy = (ny + kR - 1) / kR;
    if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
    int64_t kz_len;
    if (sizeof(T) == 8) {
        // FP64: runs of 16 planes, many waves of blocks: with about one wave
        // of long runs the blocks whose rows meet the zero faces (their
        // lanes take the FP64 fallback) finished last while SMs idled (512^3
        // step: runs of 171, 64, 32, 16, 8 planes 1.85, 1.72, 1.70, 1.70,
        // 1.71 ms with the earlier update)
        kz_len = nz < 16 ? nz : 16;
        if ((nz + kz_len - 1) / kz_len > 65535) kz_len = (nz + 65534) / 65535;
    } else {
        // split the planes into runs so that about 8 blocks per SM are in flight
        const int64_t want = (int64_t)sm_count() * 8;
        int64_t runs = (want + gx * gy - 1) / (gx * gy);
        if (runs < 1) runs = 1;
        kz_len = (nz + runs - 1) / runs;
        if (kz_len < 8) kz_len = nz < 8 ? nz : 8;
    }
    const int64_t gz = (nz + kz_len - 1) / kz_len;
    if (gz > 65535) return cudaErrorInvalidValue;
    diffuse3d_kernel<T, V><<<dim3((unsigned)gx, (unsigned)gy, (unsigned)gz), dim3(32, kR), 0,
                             stream>>>(src, dst, nx, ny, nz, alpha, kz_len);
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_steps(T *u, T *v, int64_t nx, int64_t ny, int64_t nz, T alpha, int64_t nsteps,
                         cudaStream_t stream, uint64_t *launches) {
    constexpr int VW = 16 / sizeof(T);
    const bool vec = nx % VW == 0 && (uintptr_t)u % 16 == 0 && (uintptr_t)v % 16 == 0;
    // tensor maps of both buffers (each is the source of every other step)
    CUtensorMap map_u, map_v;
    const bool bulk = sizeof(T) == 4 && vec &&
                      encode_field_map<T>(&map_u, u, nx, ny, nz) &&
                      encode_field_map<T>(&map_v, v, nx, ny, nz);
    for (int64_t s = 1; s <= nsteps; ++s) {
        const T *src = (s & 1) ? u : v;
        T *dst = (s & 1) ? v : u;
        cudaError_t e;
        if (bulk)
            e = launch_bulk<T>((s & 1) ? map_u : map_v, dst, nx, ny, nz, alpha, stream);
        else if (vec)
            e = launch_typed<T, VW>(src, dst, nx, ny, nz, alpha, stream);
        else
            e = launch_typed<T, 1>(src, dst, nx, ny, nz, alpha, stream);
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    return cudaGetLastError();
}

}  // namespace

FVF_BOUNDS_READER(read_bounds_diffuse3d)

cudaError_t read_device_error(int *flag) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_device_error, sizeof(int));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    return e;
}

cudaError_t launch_diffuse3d(void *u, void *v, int64_t nx, int64_t ny, int64_t nz, double alpha,
                             int64_t nsteps, bool fp64, cudaStream_t stream,
                             uint64_t *launches) {
    if (fp64)
        return launch_steps<double>(static_cast<double *>(u), static_cast<double *>(v), nx, ny,
                                    nz, alpha, nsteps, stream, launches);
    return launch_steps<float>(static_cast<float *>(u), static_cast<float *>(v), nx, ny, nz,
                               (float)alpha, nsteps, stream, launches);
}

}  // namespace fvf
