// Device status word shared by every kernel that has a bounded wait.
//
// A wait that gives up (a TMA copy or an MMA that never signals its mbarrier)
// writes a non-zero code here instead of trapping; sgemm_device_status() reads
// and clears it.  The word is a file-scope __device__ variable; its device
// address is looked up once per device with cudaGetSymbolAddress (no
// allocation) and passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

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

}  // namespace sgemm
