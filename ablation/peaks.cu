// peaks.cu -- issue-rate probes for the benchmark, not part of libfvf.
//
// Each probe runs independent dependency chains of one arithmetic
// instruction in every thread of a full-occupancy grid (8 blocks of 256
// threads per SM, 8 chains per thread) and reports operations per second
// from CUDA events: FP64 add, multiply and fused multiply-add, FP32 fused
// multiply-add, and a 32-bit integer xor-add pair on the ALU pipe.  The
// benchmark uses them as measured denominators for kernels bound by
// arithmetic rather than by HBM.  Built into libfvf_ablation.so with the
// ablation kernels.
#include <cuda_runtime.h>

#define ABL_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kChains = 8;
constexpr int kIters = 4096;
constexpr int kThreads = 256;

template <int OP>
__global__ void __launch_bounds__(kThreads) fp64_rate_kernel(double *out, double a, double b,
                                                             int write) {
    double x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = threadIdx.x * 1e-3 + c;
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) {
            if (OP == 0) x[c] = __dadd_rn(x[c], a);
            else if (OP == 1) x[c] = __dmul_rn(x[c], a);
            else x[c] = __fma_rn(x[c], a, b);
        }
    }
    double s = 0.0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    if (write) out[blockIdx.x * kThreads + threadIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads) fp32_rate_kernel(float *out, float a, float b,
                                                             int write) {
    float x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = threadIdx.x * 1e-3f + c;
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) x[c] = __fmaf_rn(x[c], a, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    if (write) out[blockIdx.x * kThreads + threadIdx.x] = s;
}

// two integer operations (xor, add) per chain step
__global__ void __launch_bounds__(kThreads) int_rate_kernel(unsigned *out, unsigned a,
                                                            int write) {
    unsigned x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = threadIdx.x + c;
    for (int it = 0; it < kIters; ++it) {
#pragma unroll
        for (int c = 0; c < kChains; ++c) x[c] = (x[c] ^ a) + (unsigned)c;
    }
    unsigned s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += x[c];
    if (write) out[blockIdx.x * kThreads + threadIdx.x] = s;
}

}  // namespace

// op: 0 FP64 add, 1 FP64 multiply, 2 FP64 FMA, 3 FP32 FMA, 4 integer xor+add.
// Runs one warm-up launch and `reps` timed launches on the legacy stream and
// writes the rate in operations per second (an FMA counts as one operation).
// Returns 0, or 1 for a bad argument, 2 for a CUDA error.  Synchronous.
ABL_API int bench_issue_rate(int op, int reps, double *ops_per_s) {
    if (op < 0 || op > 4 || reps < 1 || !ops_per_s) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 2;
    const int blocks = sms * 8;
    void *out = nullptr;
    if (cudaMalloc(&out, (size_t)blocks * kThreads * sizeof(double)) != cudaSuccess) return 2;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    auto launch = [&]() {
        switch (op) {
            case 0: fp64_rate_kernel<0><<<blocks, kThreads>>>((double *)out, 1.0000001, 0.5, 0); break;
            case 1: fp64_rate_kernel<1><<<blocks, kThreads>>>((double *)out, 1.0000001, 0.5, 0); break;
            case 2: fp64_rate_kernel<2><<<blocks, kThreads>>>((double *)out, 0.9999999, 1e-7, 0); break;
            case 3: fp32_rate_kernel<<<blocks, kThreads>>>((float *)out, 0.9999f, 1e-4f, 0); break;
            default: int_rate_kernel<<<blocks, kThreads>>>((unsigned *)out, 0x9E3779B9u, 0); break;
        }
    };
    launch();
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r) launch();
    cudaEventRecord(e1);
    cudaError_t e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(out);
    if (e != cudaSuccess || ms <= 0.0f) return 2;
    const double per_launch = (double)blocks * kThreads * kChains * kIters * (op == 4 ? 2 : 1);
    *ops_per_s = per_launch * reps / (ms * 1e-3);
    return 0;
}
