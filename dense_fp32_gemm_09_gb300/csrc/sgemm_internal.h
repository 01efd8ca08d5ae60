// Internal types shared by the host dispatcher and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sgemm.h"

namespace sgemm {

enum : int { kEpiPlain = 0, kEpiAlpha = 1, kEpiAlphaBeta = 2 };

// Everything one launch needs, passed by value in the kernel parameter space.
struct GemmArgs {
    int M, N, K;
    const float* A;
    const float* B;
    float* C;
    long long lda, ldb, ldc;
    int c_vec;            // 1: C and ldc allow 16-byte stores
    int epi;              // kEpiPlain (C = acc), kEpiAlpha, kEpiAlphaBeta
    float alpha, beta;    // C = alpha * A.B + beta * C (beta == 0: C is not read)

    // Tile grid and schedule (see the persistent scheduler in sgemm_ffma.cuh).
    int tiles_m, tiles_n;  // ceil(M/BM), ceil(N/BN)
    int KT;                // k-tiles per output tile: ceil(K/BK)
    int grid;              // CTAs launched (G)
    int dp_tiles;          // tiles [0, dp_tiles) are done whole by one CTA each
    int sk_tiles;          // tiles [dp_tiles, dp_tiles + sk_tiles) are split over CTAs
    long long sk_iters;    // sk_tiles * KT: k-tiles shared out over the G CTAs
    int group_m;           // tile rasterisation: tile rows per group

    float* ws_partial;     // [G][2][BM*BN] partial tiles of split tiles
    int* status;           // device status word (bounded waits that give up)
};

// One entry of the tile table.
struct KernelEntry {
    const char* name;
    const void* kernel;     // __global__ void(GemmArgs) or void(FfmaTmaParams) when tma
    int bm, bn, bk, wm, wn, tm, tn, stages, threads, smem_bytes;
    int vec;                // 4: needs 16-byte aligned A/B rows; 1: any alignment
    int fma2;
    int tma;                // 1: operands staged by TMA (tensor maps built per call)
};

// Device status word (sgemm_status.cu): address on the current device, and a
// synchronous read-and-clear of its value.
int* status_word_ptr();
int read_and_clear_status(int* value);
int run_wait_selftest(int limit_ms);

// Sums the partial tiles of a stream-K launch into C (sgemm_reduce.cu).  Launch
// it on the same stream right after the main kernel when a.sk_tiles > 0.
cudaError_t launch_sk_reduce(const GemmArgs& a, int bm, int bn, int sms, cudaStream_t stream);
int reduce_chunks(int bm, int bn, int sk_tiles, int sms);

// Sets the text sgemm_last_error() returns on this thread.
void set_last_error_message(const char* msg);

// 3xTF32 tensor-core path (sgemm_tf32x3.cu).
size_t tf32x3_workspace_bytes(int M, int N, int K);
int tf32x3_prepare(int M, int N, int K, const float* A, long long lda, const float* B,
                   long long ldb, void* ws, size_t ws_bytes, int sms, cudaStream_t stream);
int tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                    int c_vec, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                    int* launches);
int tf32x3_tile_width(int M, int N, int K, int sms);
int tf32x3_query(int M, int N, int K, int sms, sgemm_config* out);


}  // namespace sgemm
