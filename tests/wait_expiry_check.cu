// Test program for the bounded mbarrier wait (finite_volume_field_gb300/
// csrc/mbarrier.cuh): a phase that cannot complete -- a barrier expecting two
// arrivals that gets one -- must make mbar::wait give up after its poll
// limit and return false, with no copy in flight and no fault; after the
// second arrival the same wait must succeed.  Built by the GPU test with
// nvcc into a temporary directory; it launches nothing else.
#include <cuda_runtime.h>

#include "../finite_volume_field_gb300/csrc/mbarrier.cuh"

using namespace fvf;

__global__ void wait_expiry_kernel(int *status, unsigned limit) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const unsigned b = mbar::smem_addr(&bar);
    mbar::init(b, 2);
    mbar::fence_init();
    mbar::arrive(b);                                  // one of the two arrivals
    status[0] = mbar::wait(b, 0, limit) ? 1 : 2;      // must expire: 2
    mbar::arrive(b);                                  // phase 0 completes
    status[1] = mbar::wait(b, 0, limit) ? 1 : 2;      // must succeed: 1
}

extern "C" int run_wait_expiry(int *host_status, unsigned limit) {
    int *d = nullptr;
    if (cudaMalloc(&d, 2 * sizeof(int)) != cudaSuccess) return 1;
    cudaMemset(d, 0, 2 * sizeof(int));
    wait_expiry_kernel<<<1, 32>>>(d, limit);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(host_status, d, 2 * sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
