// sgemm_run_noalloc: C = A.B without any device allocation by the library.
//
// Some callers cannot let a library allocate device memory: cudaMalloc can
// synchronise the whole device and take an unbounded time, which a
// latency-critical caller cannot afford on its hot path, and processes that
// reserve their device memory budget up front must not see a library grow it
// later (or fail for lack of memory mid-run).  The split-tile (stream-K)
// schedule of sgemm_run needs scratch for partial tiles; this entry point takes
// that scratch from one fixed array compiled into the library instead of from
// a workspace it would otherwise allocate.
//
// The array is a file-scope __device__ variable.  In host code the array's
// name is only a host-side stand-in, so its device address is looked up once
// per device with cudaGetSymbolAddress (the first call on a device that needs
// scratch does this, with that device current) and passed to the kernels.
// Under CUDA's lazy module loading that lookup is what loads this file's module
// and with it reserves the array on the device; the device then holds it until
// the process exits.  sgemm_shutdown forgets the addresses (they belong to the
// primary context of each device), so the next call looks them up again.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sgemm_internal.h"

namespace sgemm {
namespace {

constexpr size_t kNoAllocScratchBytes = SGEMM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Shared by every call on a device; keeps whatever the last call wrote.  The
// kernels never read a part of it that the same call has not written first, so
// nothing in it has to start at zero.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set-up on first use).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error_message("sgemm_run_noalloc: cudaGetDevice failed");
        return SGEMM_ERR_LAUNCH;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error_message("sgemm_run_noalloc: device index out of range");
        return SGEMM_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            std::snprintf(msg, sizeof(msg),
                          "sgemm_run_noalloc: cudaGetSymbolAddress of the static scratch "
                          "failed on device %d: %s",
                          dev, cudaGetErrorString(e));
            set_last_error_message(msg);
            return SGEMM_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SGEMM_OK;
}

}  // namespace

void forget_noalloc_scratch() {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int d = 0; d < kMaxDevices; ++d) g_scratch_addr[d] = nullptr;
}

}  // namespace sgemm

extern "C" int sgemm_run_noalloc(int M, int N, int K, const float* A, int lda, const float* B,
                                 int ldb, float* C, int ldc, sgemm_stream_t stream) {
    using namespace sgemm;
    size_t need = 0;
    int rc = sgemm_workspace_size(M, N, K, lda, ldb, ldc, A, B, C, &need);
    if (rc != SGEMM_OK) return rc;
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        std::snprintf(msg, sizeof(msg),
                      "sgemm_run_noalloc: this problem needs %zu bytes of scratch; the static "
                      "scratch holds %zu bytes",
                      need, kNoAllocScratchBytes);
        set_last_error_message(msg);
        return SGEMM_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    if (need > 0) {
        rc = scratch_address(&ws);
        if (rc != SGEMM_OK) return rc;
    }
    return sgemm_run_ws(M, N, K, A, lda, B, ldb, C, ldc, ws, need, stream);
}
