// Device status word shared by every kernel that has a bounded wait.
//
// A wait that gives up (a TMA copy or an MMA that never signals its mbarrier)
// writes a non-zero code here instead of trapping; sgemm_device_status() reads
// and clears it.  The word is a file-scope __device__ variable; its device
// address is looked up once per device with cudaGetSymbolAddress (no
// allocation) and passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "sgemm_async.cuh"
#include "sgemm_internal.h"

namespace sgemm {
namespace {

__device__ int g_status_word = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_addr[kMaxDevices] = {};

}  // namespace

int* status_word_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_addr[dev] = static_cast<int*>(p);
    }
    return g_addr[dev];
}

int read_and_clear_status(int* value) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
    }
    *value = v;
    return SGEMM_OK;
}

namespace {

// One CTA waits on an mbarrier that nothing ever arrives on: the bounded wait
// must give up by itself after limit_ns and record the timeout.
__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_s;
    if (threadIdx.x == 0) {
        async::mbar_init(async::su32(&bar), 1);
        abort_s = 0;
        async::mbar_fence_init();
    }
    __syncthreads();
    async::mbar_wait(async::su32(&bar), 0, &abort_s, status, limit_ns);
}

}  // namespace

int run_wait_selftest(int limit_ms) {
    int* status = status_word_ptr();
    if (status == nullptr) return SGEMM_ERR_LAUNCH;
    wait_selftest_kernel<<<1, 32>>>(status, static_cast<unsigned long long>(limit_ms) * 1000000ull);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_OK;
}

}  // namespace sgemm
