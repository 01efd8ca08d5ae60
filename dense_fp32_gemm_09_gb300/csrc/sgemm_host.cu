// Host-buffer entry point (sgemm_run_host): the copies of A and B in, the
// product and the copy of C out, pipelined over row panels of C on three
// library-owned streams per device so that copies overlap products.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>

#include "sgemm_internal.h"

namespace sgemm {

namespace {

// ----------------------------------------------------------------------------
// Host-buffer entry: three library-owned streams per device (host-to-device
// copies, the product of each row panel of C, device-to-host copies), so that
// the copies of one panel overlap the product of another.
// ----------------------------------------------------------------------------
constexpr int kMaxHostPanels = SGEMM_HOST_MAX_PANELS;
struct HostPipe {
    int dev = 0;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t a_in[kMaxHostPanels] = {}, c_ready[kMaxHostPanels] = {};
    cudaEvent_t k_in[kMaxHostPanels] = {};   // k-chunks of the first panel
    std::mutex mu;   // one call's enqueue at a time: the events are reused
};
std::mutex g_pipe_mu;
std::map<int, HostPipe*> g_pipes;

void destroy_pipe(HostPipe* h) {
    for (cudaStream_t st : {h->h2d, h->comp, h->d2h})
        if (st) cudaStreamDestroy(st);
    for (cudaEvent_t ev : {h->start, h->done})
        if (ev) cudaEventDestroy(ev);
    for (int i = 0; i < kMaxHostPanels; ++i) {
        if (h->a_in[i]) cudaEventDestroy(h->a_in[i]);
        if (h->c_ready[i]) cudaEventDestroy(h->c_ready[i]);
        if (h->k_in[i]) cudaEventDestroy(h->k_in[i]);
    }
    delete h;
}

int host_pipe(HostPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_cuda_error("cudaGetDevice", e);
        return SGEMM_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    auto it = g_pipes.find(dev);
    if (it != g_pipes.end()) {
        *out = it->second;
        return SGEMM_OK;
    }
    HostPipe* h = new HostPipe;
    h->dev = dev;
    for (cudaStream_t* st : {&h->h2d, &h->comp, &h->d2h})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&h->start, &h->done})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int i = 0; i < kMaxHostPanels && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&h->a_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->c_ready[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->k_in[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        set_cuda_error("host pipeline streams", e);
        destroy_pipe(h);
        return SGEMM_ERR_LAUNCH;
    }
    g_pipes[dev] = h;
    *out = h;
    return SGEMM_OK;
}

// Row panels for the host-buffer entry: fills rows[] (multiples of 256 but the
// last) and returns their number.  Large problems: 25 % of the rows (computed in
// k-chunks as their inputs arrive), then 65 % in one efficient product, then a
// last 10 % whose copy back is the only exposed tail (measured best of several
// splits at 4096^3 and 8192^3); mid-size problems: two halves.  SGEMM_HOST_PANELS
// (a count of equal panels) or SGEMM_HOST_SPLIT (percentages of M, e.g.
// "25,65,10") override it (tuning).
int host_panels(int M, int N, int K, int (&rows)[kMaxHostPanels]) {
    int pct[kMaxHostPanels];
    int n_pct = 0;
    if (const char* env = std::getenv("SGEMM_HOST_SPLIT")) {
        for (const char* c = env; *c && n_pct < kMaxHostPanels;) {
            const int v = std::atoi(c);
            if (v > 0) pct[n_pct++] = v;
            while (*c && *c != ',') ++c;
            if (*c == ',') ++c;
        }
    }
    if (n_pct == 0) {
        const double macs = static_cast<double>(M) * N * K;
        if (const char* env = std::getenv("SGEMM_HOST_PANELS")) {
            n_pct = std::max(1, std::min(std::atoi(env), kMaxHostPanels));
            for (int i = 0; i < n_pct; ++i) pct[i] = 1;
        } else if (macs >= 4.0e9) {
            n_pct = 3;
            pct[0] = 25;
            pct[1] = 65;
            pct[2] = 10;
        } else {
            n_pct = macs >= 5.0e8 ? 2 : 1;
            for (int i = 0; i < n_pct; ++i) pct[i] = 1;
        }
    }
    long long total = 0;
    for (int i = 0; i < n_pct; ++i) total += pct[i];
    int n = 0, done = 0;
    for (int i = 0; i < n_pct && done < M; ++i) {
        // Panels of whole 256-row tiles (two 128-row ones): a panel that ends
        // inside a tile row computes the rest of that row for nothing.
        int r = static_cast<int>(M * static_cast<long long>(pct[i]) / total);
        r = std::max(256, (r + 128) / 256 * 256);
        if (i == n_pct - 1 || done + r > M) r = M - done;
        rows[n++] = r;
        done += r;
    }
    return n;
}

// Depth of the k-chunks in which the first row panel is computed, so that its
// product starts after one chunk of A and B has arrived rather than all of B;
// K when it is not chunked.  SGEMM_HOST_KCHUNKS overrides (tuning).
int host_kchunk(int M, int N, int K) {
    int chunks = 1;
    if (const char* env = std::getenv("SGEMM_HOST_KCHUNKS")) {
        chunks = std::atoi(env);
    } else {
        const double macs = static_cast<double>(M) * N * K;
        chunks = macs >= 4.0e9 ? 4 : (macs >= 5.0e8 ? 2 : 1);
    }
    chunks = std::max(1, std::min(chunks, kMaxHostPanels));
    const int depth = ((K + chunks - 1) / chunks + 63) / 64 * 64;
    return std::min(K, std::max(64, depth));
}

}  // namespace

void shutdown_host_pipes() {
    std::lock_guard<std::mutex> lp(g_pipe_mu);
    for (auto& kv : g_pipes) {
        int prev = 0;
        cudaGetDevice(&prev);
        cudaSetDevice(kv.first);
        destroy_pipe(kv.second);
        cudaSetDevice(prev);
    }
    g_pipes.clear();
}

}  // namespace sgemm

using namespace sgemm;

extern "C" {

int sgemm_host_plan_check(int M, int N, int K, int* n_panels, int* rows, int* k_chunk) {
    if (M <= 0 || N <= 0 || K < 0 || n_panels == nullptr) return SGEMM_ERR_INVALID_ARG;
    if (check_sizes(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    int r[kMaxHostPanels];
    const int n = host_panels(M, N, K, r);
    *n_panels = n;
    if (rows)
        for (int i = 0; i < n; ++i) rows[i] = r[i];
    if (k_chunk) *k_chunk = K > 0 ? host_kchunk(M, N, K) : 0;
    return SGEMM_OK;
}

int sgemm_run_host(int M, int N, int K, const float* hA, int lda, const float* hB, int ldb,
                   float* hC, int ldc, float* dA, float* dB, float* dC, sgemm_stream_t stream) {
    int rc = check_operands(0, 0, M, N, K, hA, lda, hB, ldb, hC, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (dC == nullptr || (K > 0 && (dA == nullptr || dB == nullptr))) {
        set_last_error_message("null device buffer");
        return SGEMM_ERR_INVALID_ARG;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rows[kMaxHostPanels];
    const int n_panels = host_panels(M, N, K, rows);
    const size_t fa = sizeof(float) * lda, fb = sizeof(float) * ldb, fc = sizeof(float) * ldc;
    if (n_panels == 1) {
        // One panel: nothing to overlap, so the copies and the product are queued on
        // `stream` itself, without the library streams' fork and join (256^3: 24.3
        // against 25.0 us a call; the copies' own latency is the rest).
        cudaError_t e = cudaSuccess;
        if (K > 0) {
            e = cudaMemcpy2DAsync(dA, fa, hA, fa, sizeof(float) * K, M,
                                  cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess)
                e = cudaMemcpy2DAsync(dB, fb, hB, fb, sizeof(float) * N, K,
                                      cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) {
                set_cuda_error("host-to-device copy", e);
                return SGEMM_ERR_LAUNCH;
            }
        }
        rc = sgemm_run(M, N, K, K > 0 ? dA : nullptr, lda, K > 0 ? dB : nullptr, ldb, dC, ldc,
                       stream);
        if (rc != SGEMM_OK) return rc;
        e = cudaMemcpy2DAsync(hC, fc, dC, fc, sizeof(float) * N, M, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) {
            set_cuda_error("device-to-host copy", e);
            return SGEMM_ERR_LAUNCH;
        }
        return SGEMM_OK;
    }
    HostPipe* hp = nullptr;
    rc = host_pipe(&hp);
    if (rc != SGEMM_OK) return rc;
    std::lock_guard<std::mutex> lk(hp->mu);
    // Fork: the three streams start after the work already queued on `s`.
    cudaError_t e = cudaEventRecord(hp->start, s);
    for (cudaStream_t st : {hp->h2d, hp->comp, hp->d2h})
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp->start, 0);
    if (e != cudaSuccess) {
        set_cuda_error("host pipeline fork", e);
        return SGEMM_ERR_LAUNCH;
    }
    const char* failed = nullptr;
    const int kc = host_kchunk(M, N, K);
    if (K > 0) {
        // Copy order: the first panel's A and B k-chunk by k-chunk (all of B
        // once the last chunk is in), then the other panels' A.
        const int mr0 = rows[0];
        for (int c = 0, k0 = 0; k0 < K && e == cudaSuccess; ++c, k0 += kc) {
            const int kw = std::min(kc, K - k0);
            const long long ob = static_cast<long long>(k0) * ldb;
            e = cudaMemcpy2DAsync(dA + k0, fa, hA + k0, fa, sizeof(float) * kw, mr0,
                                  cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess)
                e = cudaMemcpy2DAsync(dB + ob, fb, hB + ob, fb, sizeof(float) * N, kw,
                                      cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess) e = cudaEventRecord(hp->k_in[c], hp->h2d);
        }
        for (int p = 1, r0 = rows[0]; p < n_panels && e == cudaSuccess; r0 += rows[p++]) {
            const long long oa = static_cast<long long>(r0) * lda;
            e = cudaMemcpy2DAsync(dA + oa, fa, hA + oa, fa, sizeof(float) * K, rows[p],
                                  cudaMemcpyHostToDevice, hp->h2d);
            if (e == cudaSuccess) e = cudaEventRecord(hp->a_in[p], hp->h2d);
        }
        if (e != cudaSuccess) failed = "host-to-device copy";
    }
    for (int p = 0, r0 = 0; p < n_panels && failed == nullptr && rc == SGEMM_OK;
         r0 += rows[p++]) {
        const int mr = rows[p];
        const long long oa = static_cast<long long>(r0) * lda;
        const long long oc = static_cast<long long>(r0) * ldc;
        const sgemm_stream_t comp = reinterpret_cast<sgemm_stream_t>(hp->comp);
        if (K == 0) {
            rc = sgemm_run(mr, N, 0, nullptr, lda, nullptr, ldb, dC + oc, ldc, comp);
        } else if (p == 0) {
            // C_panel = sum over chunks of A[:, chunk] . B[chunk, :], in order.
            for (int c = 0, k0 = 0; k0 < K && rc == SGEMM_OK; ++c, k0 += kc) {
                e = cudaStreamWaitEvent(hp->comp, hp->k_in[c], 0);
                if (e != cudaSuccess) {
                    failed = "host pipeline wait";
                    break;
                }
                rc = sgemm_run_ex(mr, N, std::min(kc, K - k0), 1.0f, dA + k0, lda,
                                  dB + static_cast<long long>(k0) * ldb, ldb,
                                  k0 == 0 ? 0.0f : 1.0f, dC + oc, ldc, -1, 0, comp);
            }
        } else {
            e = cudaStreamWaitEvent(hp->comp, hp->a_in[p], 0);
            if (e != cudaSuccess) {
                failed = "host pipeline wait";
                break;
            }
            rc = sgemm_run(mr, N, K, dA + oa, lda, dB, ldb, dC + oc, ldc, comp);
        }
        if (rc != SGEMM_OK || failed != nullptr) break;
        e = cudaEventRecord(hp->c_ready[p], hp->comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->c_ready[p], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(hC + oc, fc, dC + oc, fc, sizeof(float) * N, mr,
                                  cudaMemcpyDeviceToHost, hp->d2h);
        if (e != cudaSuccess) failed = "device-to-host copy";
    }
    const cudaError_t fail_e = e;
    // Join: `s` continues once the last panel is back, which on success follows
    // every copy and product of this call.  After a failure part of the
    // pipeline may not lead to that copy (copies in of later panels, say), so
    // the other two streams are joined as well.  A wait uses the event as last
    // recorded when the wait is issued, so `done` serves all three.
    cudaError_t j = cudaSuccess;
    if (failed != nullptr || rc != SGEMM_OK) {
        for (cudaStream_t st : {hp->h2d, hp->comp}) {
            if (j == cudaSuccess) j = cudaEventRecord(hp->done, st);
            if (j == cudaSuccess) j = cudaStreamWaitEvent(s, hp->done, 0);
        }
    }
    if (j == cudaSuccess) j = cudaEventRecord(hp->done, hp->d2h);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(s, hp->done, 0);
    if (failed != nullptr) {
        set_cuda_error(failed, fail_e);
        return SGEMM_ERR_LAUNCH;
    }
    if (rc != SGEMM_OK) return rc;
    if (j != cudaSuccess) {
        set_cuda_error("host pipeline join", j);
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

}  // extern "C"
