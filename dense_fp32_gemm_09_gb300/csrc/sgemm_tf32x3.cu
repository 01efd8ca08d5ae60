// 3xTF32 tensor-core SGEMM on sm_103a (tcgen05 + TMEM + TMA).
//
// The product the pages compute ("Register/Shared Memory Tiling", 관련 개념 and
// 장단점 #3 point at pairing the tile hierarchy with tensor-core MMA) is run on
// the 5th-generation tensor cores while keeping FP32-level accuracy: every
// operand is split into two TF32 numbers, x = hi + lo with
//     hi = x with its 13 low mantissa bits cleared   (exact in TF32)
//     lo = round_to_tf32(x - hi)                       (x - hi is exact in fp32)
// and  A.B ~= Ahi.Bhi + Ahi.Blo + Alo.Bhi  (the Alo.Blo term, ~2^-22 relative,
// is dropped).  Each product of two TF32 numbers is exact in fp32 and the three
// MMAs accumulate in fp32 in tensor memory.
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   * split_a_kernel / split_bt_kernel write Ahi, Alo (M x Kp, K-major like A)
//     and Bhi^T, Blo^T (N x Kp, K-major: B transposed) to a workspace;
//   * warp 0, one thread: TMA loads of the four K-major 128-byte-swizzled tiles
//     of a k-block into a STAGES-deep ring, signalled through mbarriers;
//   * warp 1, one thread: allocates tensor memory and issues
//     tcgen05.mma.kind::tf32 (M = 128, N = BN, K = 8) into one of two fp32
//     accumulators in TMEM; tcgen05.commit releases smem stages and hands a
//     finished accumulator to the epilogue;
//   * warps 2..5: read the accumulator with tcgen05.ld (each warp its 32 TMEM
//     lanes = 32 rows of the tile) and store C, then free the accumulator.
// Every mbarrier wait is bounded in time; a wait that gives up writes the
// library's device status word (read by sgemm_device_status) and the CTA drains
// and exits instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "sgemm_async.cuh"
#include "sgemm_internal.h"

namespace sgemm {
namespace tc {

using async::gtimer;
using async::mbar_arrive;
using async::mbar_expect_tx;
using async::mbar_init;
using async::su32;
using async::tma_load_2d;

constexpr int BM = 128;
constexpr int BK = 32;        // fp32 per k-block row: one 128-byte swizzle row
constexpr int UMMA_K = 8;     // K of one tcgen05.mma .kind::tf32
// warp 0: TMA, warp 1: MMA, then 4 epilogue warps per 128 accumulator columns
__host__ __device__ constexpr int tf32x3_threads(int bn) { return 64 + 32 * 4 * (bn / 128); }

// Workspace regions are padded to 256 bytes (TMA wants 16-byte aligned bases).
inline size_t align_up_floats(size_t n) { return (n + 63) / 64 * 64; }

struct Params {
    CUtensorMap tm_ahi, tm_alo, tm_bhi, tm_blo;
    float* C;
    long long ldc;
    int M, N, K;
    int tiles_m, tiles_n, kblocks;
    int c_vec;
    int epi;
    float alpha, beta;
    int* status;      // device status word for waits that give up
};

// ----------------------------------------------------------------------------
// PTX wrappers
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with
// 128-byte swizzling: rows of 128 bytes, the swizzle pattern repeating every 8
// rows (1024 bytes = the stride between 8-row groups), one swizzle atom along K.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address
    d |= static_cast<uint64_t>(0) << 16;                      // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t tf32_idesc(int bn) {
    return (1u << 4)                                   // D format: f32
           | (2u << 7)                                 // A format: tf32
           | (2u << 10)                                // B format: tf32
           | (static_cast<uint32_t>(bn >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(BM >> 4) << 24);   // M / 16
}

// Tile index -> origin: groups of 8 tile rows, column-major inside a group, so
// CTAs running together share A rows and B columns in L2.
__device__ __forceinline__ void tile_mn(const Params& p, int tile, int bn, int& m0, int& n0) {
    const int gm = 8;
    const int group_size = gm * p.tiles_n;
    const int group = tile / group_size;
    const int first_m = group * gm;
    const int rows = min(p.tiles_m - first_m, gm);
    const int r = tile - group * group_size;
    m0 = (first_m + r % rows) * BM;
    n0 = (r / rows) * bn;
}

__device__ __forceinline__ float epi_one(const Params& p, float acc, const float* c) {
    if (p.epi == kEpiPlain) return acc;
    if (p.epi == kEpiAlpha) return p.alpha * acc;
    return fmaf(p.alpha, acc, p.beta * *c);
}

// The tensor core adds products into its fp32 accumulator with truncation, so
// summing a long K range in one TMEM accumulator biases the result by about
// (K / 8) x 3 x half an ulp of |C|.  The K range of a tile is therefore cut into
// chunks of KC_BLOCKS k-blocks: each chunk is accumulated in TMEM from zero, and
// the epilogue warps add the finished chunk into an fp32 running sum in
// registers with round-to-nearest adds.  Two TMEM chunk buffers alternate so the
// MMAs of chunk c+1 overlap the epilogue's read of chunk c.
template <int BN, int STAGES, int KC_BLOCKS>
__global__ void __launch_bounds__(tf32x3_threads(BN), 1)
    tf32x3_kernel(const __grid_constant__ Params p) {
    constexpr int EPI_WARPS = 4 * (BN / 128);
    constexpr uint32_t A_BYTES = BM * BK * 4;
    constexpr uint32_t B_BYTES = BN * BK * 4;
    constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * BN;   // two chunk accumulators
    static_assert(BN == 128 || BN == 256, "BN");
    static_assert(TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512,
                  "TMEM allocation must be a power of two");

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem0 = su32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = p.tiles_m * p.tiles_n;
    const int chunks = (p.kblocks + KC_BLOCKS - 1) / KC_BLOCKS;
    volatile int* abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(su32(&full_bar[s]), 1);
            mbar_init(su32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(su32(&tfull_bar[b]), 1);
            mbar_init(su32(&tempty_bar[b]), EPI_WARPS);
        }
        abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&tmem_base_s)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[STAGES];
            bool issued[STAGES];
            for (int s = 0; s < STAGES; ++s) issued[s] = false;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                int m0, n0;
                tile_mn(p, tile, BN, m0, n0);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!async::mbar_wait(su32(&empty_bar[stage]), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = su32(&full_bar[stage]);
                    const uint32_t base = smem0 + stage * STAGE_BYTES;
                    mbar_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(base, &p.tm_ahi, kb * BK, m0, fb);
                    tma_load_2d(base + A_BYTES, &p.tm_alo, kb * BK, m0, fb);
                    tma_load_2d(base + 2 * A_BYTES, &p.tm_bhi, kb * BK, n0, fb);
                    tma_load_2d(base + 2 * A_BYTES + B_BYTES, &p.tm_blo, kb * BK, n0, fb);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Aborting: let copies already in flight land before the CTA exits.
                volatile int no_abort = 0;
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s]) async::mbar_wait(su32(&full_bar[s]), issued_phase[s], &no_abort, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = tf32_idesc(BN);
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                for (int c = 0; ok && c < chunks; ++c) {
                    if (!async::mbar_wait(su32(&tempty_bar[buf]), buf_phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                    const int kb_end = min(p.kblocks, (c + 1) * KC_BLOCKS);
                    for (int kb = c * KC_BLOCKS; kb < kb_end; ++kb) {
                        if (!async::mbar_wait(su32(&full_bar[stage]), phase, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t base = smem0 + stage * STAGE_BYTES;
                        const bool first = (kb == c * KC_BLOCKS);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint32_t off = k * UMMA_K * 4;
                            const uint64_t ahi = sw128_kmajor_desc(base + off);
                            const uint64_t alo = sw128_kmajor_desc(base + A_BYTES + off);
                            const uint64_t bhi = sw128_kmajor_desc(base + 2 * A_BYTES + off);
                            const uint64_t blo =
                                sw128_kmajor_desc(base + 2 * A_BYTES + B_BYTES + off);
                            umma_tf32(d_tmem, alo, bhi, idesc, (first && k == 0) ? 0u : 1u);
                            umma_tf32(d_tmem, ahi, blo, idesc, 1u);
                            umma_tf32(d_tmem, ahi, bhi, idesc, 1u);
                        }
                        umma_commit(su32(&empty_bar[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(su32(&tfull_bar[buf]));
                    buf ^= 1;
                    if (buf == 0) buf_phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------- epilogue: TMEM chunks -> fp32 sums -> C ----------------
        // Warp w may read TMEM lanes [32 (w % 4), +32) = 32 rows of the tile; the
        // epilogue warps come in groups of four, group g owning columns
        // [128 g, 128 g + 128).
        constexpr int EC = 128;            // accumulator columns per epilogue warp
        const int q = warp & 3;
        const int col0 = EC * ((warp - 2) / 4);
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
            int m0, n0;
            tile_mn(p, tile, BN, m0, n0);
            float sum[EC];
#pragma unroll
            for (int i = 0; i < EC; ++i) sum[i] = 0.0f;
            for (int c = 0; c < chunks; ++c) {
                if (!async::mbar_wait(su32(&tfull_bar[buf]), buf_phase, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < EC / 32; ++j) {
                    float v[32];
                    __syncwarp();   // tcgen05.ld is warp-collective
                    tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                  static_cast<uint32_t>(buf * BN + col0 + 32 * j),
                              v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sum[32 * j + i] += v[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(su32(&tempty_bar[buf]));
                buf ^= 1;
                if (buf == 0) buf_phase ^= 1u;
            }
            if (!ok) break;
            const int row = m0 + 32 * q + lane;
            if (row < p.M) {
                float* crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
                for (int j = 0; j < EC / 32; ++j) {
                    const int c0 = n0 + col0 + 32 * j;
                    if (p.c_vec && c0 + 31 < p.N) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float4 o = make_float4(sum[32 * j + 4 * u], sum[32 * j + 4 * u + 1],
                                                   sum[32 * j + 4 * u + 2],
                                                   sum[32 * j + 4 * u + 3]);
                            if (p.epi != kEpiPlain) {
                                const float* cp = crow + c0 + 4 * u;
                                o.x = epi_one(p, o.x, cp + 0);
                                o.y = epi_one(p, o.y, cp + 1);
                                o.z = epi_one(p, o.z, cp + 2);
                                o.w = epi_one(p, o.w, cp + 3);
                            }
                            *reinterpret_cast<float4*>(crow + c0 + 4 * u) = o;
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            if (c0 + u < p.N)
                                crow[c0 + u] = epi_one(p, sum[32 * j + u], crow + c0 + u);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ----------------------------------------------------------------------------
// Operand split: x -> (hi, lo) TF32 pair, A kept K-major, B transposed to K-major
// ----------------------------------------------------------------------------
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x - hi));
    lo = __uint_as_float(r);
}

// Ahi/Alo[i*Kp + k] for i < M, k < Kp (zeros for K <= k < Kp).  Each thread
// writes 4 consecutive k of one row as one float4 of hi and one of lo; it reads
// A with a float4 too when the row is 16-byte aligned (vec_in) and whole.
__global__ void __launch_bounds__(256) split_a_kernel(const float* __restrict__ A, long long lda,
                                                      int M, int K, int Kp, int vec_in,
                                                      float* __restrict__ hi,
                                                      float* __restrict__ lo) {
    const int k = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (k >= Kp) return;
    for (int i = blockIdx.y; i < M; i += gridDim.y) {
        const float* arow = A + static_cast<long long>(i) * lda;
        float x[4];
        if (vec_in && k + 3 < K) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(arow + k));
            x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = (k + u < K) ? __ldg(arow + k + u) : 0.0f;
        }
        float h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) split_tf32(x[u], h[u], l[u]);
        const long long o = static_cast<long long>(i) * Kp + k;
        *reinterpret_cast<float4*>(hi + o) = make_float4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<float4*>(lo + o) = make_float4(l[0], l[1], l[2], l[3]);
    }
}

// Bhi/Blo[n*Kp + k] = split(B[k*ldb + n]) for n < N, k < Kp, through a 64 x 64
// shared tile: reads along n and writes along k, both as float4 (reads fall back
// to scalars when B's rows are not 16-byte aligned).
constexpr int kTT = 64;
__global__ void __launch_bounds__(256) split_bt_kernel(const float* __restrict__ B, long long ldb,
                                                       int K, int N, int Kp, int vec_in,
                                                       float* __restrict__ hi,
                                                       float* __restrict__ lo) {
    __shared__ float th[kTT][kTT + 1];
    __shared__ float tl[kTT][kTT + 1];
    const int k0 = blockIdx.y * kTT, n0 = blockIdx.x * kTT;
    const int c4 = (threadIdx.x & 15) * 4;   // 16 threads x 4 columns per row
    const int r0 = threadIdx.x >> 4;         // 16 rows per pass
#pragma unroll
    for (int pass = 0; pass < kTT / 16; ++pass) {
        const int r = r0 + 16 * pass;        // k within the tile
        const int k = k0 + r, n = n0 + c4;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (k < K) {
            const float* brow = B + static_cast<long long>(k) * ldb;
            if (vec_in && n + 3 < N) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(brow + n));
                x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) x[u] = (n + u < N) ? __ldg(brow + n + u) : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) split_tf32(x[u], th[r][c4 + u], tl[r][c4 + u]);
    }
    __syncthreads();
#pragma unroll
    for (int pass = 0; pass < kTT / 16; ++pass) {
        const int nr = r0 + 16 * pass;       // n within the tile
        const int n = n0 + nr, k = k0 + c4;
        if (n < N && k < Kp) {
            const long long o = static_cast<long long>(n) * Kp + k;
            *reinterpret_cast<float4*>(hi + o) =
                make_float4(th[c4][nr], th[c4 + 1][nr], th[c4 + 2][nr], th[c4 + 3][nr]);
            *reinterpret_cast<float4*>(lo + o) =
                make_float4(tl[c4][nr], tl[c4 + 1][nr], tl[c4 + 2][nr], tl[c4 + 3][nr]);
        }
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
constexpr int kChunkBlocks = 4;   // 128 of K per TMEM chunk
// Two output-tile widths: 128 columns with 3 pipeline stages, or 256 columns
// with 2 (the shared-memory ring holds 192 KB either way).
template <int BN>
struct Variant {
    static constexpr int kStages = BN == 256 ? 2 : 3;
    static constexpr int kThreads = tf32x3_threads(BN);
    static constexpr size_t kSmem =
        static_cast<size_t>(kStages) * (2 * BM * BK * 4 + 2 * BN * BK * 4) + 1024;
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// rows x K fp32 matrix with row pitch Kp floats; box = 32 (K) x box_rows.
bool encode_kmajor(CUtensorMap* tm, const float* base, int rows, int K, int Kp, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(Kp) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t region_floats(long long rows, int Kp) {
    return align_up_floats(static_cast<size_t>(rows) * Kp);
}

}  // namespace tc

size_t tf32x3_workspace_bytes(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int Kp = (K + 3) / 4 * 4;
    return 4 * (2 * tc::region_floats(M, Kp) + 2 * tc::region_floats(N, Kp));
}

namespace {
struct WsLayout {
    float *ahi, *alo, *bhi, *blo;
};
WsLayout ws_layout(void* ws, int M, int N, int Kp) {
    WsLayout L;
    L.ahi = static_cast<float*>(ws);
    L.alo = L.ahi + tc::region_floats(M, Kp);
    L.bhi = L.alo + tc::region_floats(M, Kp);
    L.blo = L.bhi + tc::region_floats(N, Kp);
    return L;
}
}  // namespace

int tf32x3_prepare(int M, int N, int K, const float* A, long long lda, const float* B,
                   long long ldb, void* ws, size_t ws_bytes, int sms, cudaStream_t stream) {
    using namespace tc;
    if (ws == nullptr || ws_bytes < tf32x3_workspace_bytes(M, N, K)) {
        set_last_error_message("tf32x3: workspace too small");
        return SGEMM_ERR_WORKSPACE;
    }
    const int Kp = (K + 3) / 4 * 4;
    const WsLayout L = ws_layout(ws, M, N, Kp);
    (void)sms;
    if ((Kp + kTT - 1) / kTT > 65535) {
        set_last_error_message("tf32x3: K too large for the split kernels' grid");
        return SGEMM_ERR_UNSUPPORTED;
    }
    const int a_vec = ((reinterpret_cast<uintptr_t>(A) & 15) == 0 && lda % 4 == 0) ? 1 : 0;
    const int b_vec = ((reinterpret_cast<uintptr_t>(B) & 15) == 0 && ldb % 4 == 0) ? 1 : 0;
    const dim3 ga((Kp / 4 + 255) / 256, std::min(M, 65535));
    split_a_kernel<<<ga, 256, 0, stream>>>(A, lda, M, K, Kp, a_vec, L.ahi, L.alo);
    const dim3 gb((N + kTT - 1) / kTT, (Kp + kTT - 1) / kTT);
    split_bt_kernel<<<gb, 256, 0, stream>>>(B, ldb, K, N, Kp, b_vec, L.bhi, L.blo);
    if (cudaGetLastError() != cudaSuccess) {
        set_last_error_message("tf32x3: split kernels failed to launch");
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

namespace {

// Fraction of the last wave of `tiles` tiles over `ctas` CTAs that does work.
double wave_efficiency(long long tiles, int ctas) {
    const long long waves = (tiles + ctas - 1) / ctas;
    return static_cast<double>(tiles) / static_cast<double>(waves * ctas);
}

template <int BN>
int launch_variant(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                   int c_vec, const WsLayout& L, int Kp, int sms, cudaStream_t stream) {
    using namespace tc;
    using V = Variant<BN>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(tf32x3_kernel<BN, V::kStages, kChunkBlocks>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(V::kSmem));
    });
    if (attr_err != cudaSuccess) {
        set_last_error_message("tf32x3: cannot set the kernel's shared-memory size");
        return SGEMM_ERR_LAUNCH;
    }
    Params p{};
    if (!encode_kmajor(&p.tm_ahi, L.ahi, M, K, Kp, BM) ||
        !encode_kmajor(&p.tm_alo, L.alo, M, K, Kp, BM) ||
        !encode_kmajor(&p.tm_bhi, L.bhi, N, K, Kp, BN) ||
        !encode_kmajor(&p.tm_blo, L.blo, N, K, Kp, BN)) {
        set_last_error_message("tf32x3: cuTensorMapEncodeTiled failed");
        return SGEMM_ERR_LAUNCH;
    }
    p.C = C;
    p.ldc = ldc;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.kblocks = (K + BK - 1) / BK;
    p.c_vec = c_vec;
    p.alpha = alpha;
    p.beta = beta;
    p.epi = (beta != 0.0f) ? kEpiAlphaBeta : (alpha != 1.0f ? kEpiAlpha : kEpiPlain);
    p.status = status_word_ptr();
    const int tiles = p.tiles_m * p.tiles_n;
    const int grid = std::min(tiles, sms);
    tf32x3_kernel<BN, V::kStages, kChunkBlocks><<<grid, V::kThreads, V::kSmem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) {
        set_last_error_message("tf32x3: GEMM kernel failed to launch");
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

}  // namespace

int tf32x3_tile_width(int M, int N, int sms) {
    if (const char* force = std::getenv("SGEMM_TF32X3_BN")) {
        const int bn = std::atoi(force);
        if (bn == 128 || bn == 256) return bn;
    }
    // 256-wide tiles run about 5 % faster per tile (each MMA re-reads A for twice
    // the columns) but quantise into fewer, larger waves and pad narrow C more:
    // pick the better expected efficiency.
    const long long tm = (M + tc::BM - 1) / tc::BM;
    const long long t128 = (N + 127) / 128, t256 = (N + 255) / 256;
    const double e128 = wave_efficiency(tm * t128, sms) * N / (128.0 * t128);
    const double e256 = wave_efficiency(tm * t256, sms) * N / (256.0 * t256);
    return e256 * 1.05 > e128 ? 256 : 128;
}

int tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                    int c_vec, void* ws, size_t ws_bytes, int sms, cudaStream_t stream) {
    if (ws == nullptr || ws_bytes < tf32x3_workspace_bytes(M, N, K)) {
        set_last_error_message("tf32x3: workspace too small");
        return SGEMM_ERR_WORKSPACE;
    }
    const int Kp = (K + 3) / 4 * 4;
    const WsLayout L = ws_layout(ws, M, N, Kp);
    if (tf32x3_tile_width(M, N, sms) == 256)
        return launch_variant<256>(M, N, K, alpha, beta, C, ldc, c_vec, L, Kp, sms, stream);
    return launch_variant<128>(M, N, K, alpha, beta, C, ldc, c_vec, L, Kp, sms, stream);
}

}  // namespace sgemm
