// Types the kernels see: the launch arguments (passed by value in the kernel
// parameter space), the epilogue modes and one tile-table record.
#pragma once

#include <stdint.h>

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
    int sk_gap;            // virtual k-tiles counted between split tiles (sgemm_sched.cuh)
    int group_m;           // tile rasterisation: tile rows per group
    int cl_split;          // > 1: every tile is split over a cluster of cl_split CTAs
                           // that sum their partials in distributed shared memory

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

}  // namespace sgemm
