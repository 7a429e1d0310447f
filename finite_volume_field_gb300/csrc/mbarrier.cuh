// mbarrier.cuh -- shared-memory mbarrier and bulk-copy helpers (inline PTX,
// sm_90 and later) for kernels that stage data with the copy engine.
//
// Every wait is bounded: mbar_wait polls try_wait at most `limit` times and
// returns false if the phase has not completed by then, so a kernel never
// spins forever on a copy that does not land; the caller decides what to do
// (record an error, let its copies in flight finish, return).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fvf {
namespace mbar {

constexpr uint32_t kWaitLimit = 1u << 22;  // default number of try_wait polls

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the copy engine.
__device__ __forceinline__ void fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival that also expects `bytes` more bytes of copies on this phase.
__device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity to complete; false if `limit`
// polls pass first.
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity,
                                     uint32_t limit = kWaitLimit) {
    for (uint32_t it = 0; it < limit; ++it)
        if (try_wait(bar, parity)) return true;
    return false;
}

// One box of a 3D tensor map at (x, y, z) into shared memory (128-byte
// aligned), completion counted on `bar`.
__device__ __forceinline__ void tensor_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                               int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

}  // namespace mbar
}  // namespace fvf
