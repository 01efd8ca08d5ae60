// mbarrier and TMA (cp.async.bulk.tensor) wrappers shared by the TMA-fed kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace sgemm {
namespace async {

constexpr unsigned long long kWaitNs = 4000000000ull;  // a wait gives up after 4 s
constexpr unsigned kMaxSpins = 1u << 30;                // ... or this many polls
constexpr int kStatusWaitTimeout = 1;                    // code written to the status word

__device__ __forceinline__ uint32_t su32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase of `bar` with parity `parity`.  Gives up (returns false)
// when *abort is set by another thread, or after kWaitNs / kMaxSpins; then it
// records kStatusWaitTimeout in *status (if given) and sets *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status,
                                          unsigned long long limit_ns = kWaitNs) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = gtimer();
    for (unsigned i = 1; i < kMaxSpins; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (gtimer() - t0 > limit_ns) break;
        }
    }
    if (status) atomicExch(status, kStatusWaitTimeout);
    *abort = 1;
    return false;
}
// 2-D tiled TMA load of the box at (x, y) (x innermost) into shared memory at
// `dst`, completing on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

}  // namespace async
}  // namespace sgemm
