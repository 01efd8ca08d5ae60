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
// Structure (one CTA per SM, persistent; the same data-parallel + stream-K
// schedule as the FFMA kernels, over 128 x BN output tiles and 32-deep k-blocks):
//   * split_kernel (one launch) writes Ahi, Alo (M x Kp, K-major like A) and
//     Bhi^T, Blo^T (N x Kp, K-major: B transposed) to a workspace;
//   * warp 0, one thread: TMA loads of the four K-major 128-byte-swizzled tiles
//     of a k-block into a STAGES-deep ring, signalled through mbarriers;
//   * warp 1, one thread: allocates tensor memory and issues
//     tcgen05.mma.kind::tf32 (M = 128, N = BN, K = 8) into one of two fp32
//     accumulators in TMEM; tcgen05.commit releases smem stages and hands a
//     finished accumulator to the epilogue;
//   * warps 2..5 (2..9 for BN = 256): read the accumulator with tcgen05.ld (each
//     warp its 32 TMEM lanes = 32 rows of the tile), then free it; a tile whose
//     whole K range this CTA ran is stored to C, a stream-K part of a split tile
//     to the CTA's partial slot, summed into C by sk_reduce_kernel afterwards.
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
#include <vector>

#include "sgemm_async.cuh"
#include "sgemm_epilogue.cuh"
#include "sgemm_internal.h"
#include "sgemm_sched.cuh"
#include "sgemm_tma_host.h"

namespace sgemm {
namespace tc {

using async::gtimer;
using async::mbar_arrive;
using async::mbar_expect_tx;
using async::mbar_init;
using async::su32;
using async::tma_load_2d;

constexpr int BM = 128;
constexpr int UMMA_K = 8;     // K of one tcgen05.mma .kind::tf32
constexpr int KCHUNK = 128;   // K accumulated per TMEM chunk (see the kernel)
// warp 0: TMA, warp 1: MMA, then 4 epilogue warps per 128 accumulator columns
__host__ __device__ constexpr int tf32x3_threads(int bn) { return 64 + 32 * 4 * (bn / 128); }

// Workspace regions are padded to 256 bytes (TMA wants 16-byte aligned bases).
inline size_t align_up_floats(size_t n) { return (n + 63) / 64 * 64; }

struct Params {
    CUtensorMap tm_ahi, tm_alo, tm_bhi, tm_blo;
    // C, its epilogue, the persistent / stream-K schedule (k-blocks of BKT), the
    // partial-tile workspace and the device status word; A and B are unused.
    GemmArgs s;
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
// the swizzle matching its row width: BKT fp32 of K per row (32 -> 128-byte rows,
// 128-byte swizzle; 16 -> 64-byte rows, 64-byte swizzle), the pattern repeating
// every 8 rows (8 rows x row bytes = the stride between 8-row groups), one
// swizzle atom along K.
template <int BKT>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) {
    static_assert(BKT == 32 || BKT == 16, "k-block depth");
    constexpr uint64_t kRowBytes = BKT * 4;
    constexpr uint64_t kLayout = BKT == 32 ? 2 : 4;           // 128-byte / 64-byte swizzle
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address
    d |= static_cast<uint64_t>(0) << 16;                      // leading byte offset (unused)
    d |= ((8 * kRowBytes) >> 4) << 32;                        // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
    d |= kLayout << 61;                                       // swizzle mode
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

constexpr int kStageFloats = 32 * 32;   // epilogue staging block of one warp

// The tensor core adds products into its fp32 accumulator with truncation, so
// summing a long K range in one TMEM accumulator biases the result by about
// (K / 8) x 3 x half an ulp of |C|.  The K range of a tile is therefore cut into
// chunks of KC_BLOCKS k-blocks: each chunk is accumulated in TMEM from zero, and
// the epilogue warps add the finished chunk into an fp32 running sum in
// registers with round-to-nearest adds.  Two TMEM chunk buffers alternate so the
// MMAs of chunk c+1 overlap the epilogue's read of chunk c.  Chunk boundaries
// are the multiples of KC_BLOCKS k-blocks (and the ends of a CTA's part of a
// tile), so a tile computed whole is chunked the same way under any schedule.
template <int BN, int BKT, int STAGES>
__global__ void __launch_bounds__(tf32x3_threads(BN), 1)
    tf32x3_kernel(const __grid_constant__ Params p) {
    constexpr int EPI_WARPS = 4 * (BN / 128);
    constexpr int KC_BLOCKS = KCHUNK / BKT;   // k-blocks per TMEM chunk
    constexpr uint32_t A_BYTES = BM * BKT * 4;
    constexpr uint32_t B_BYTES = BN * BKT * 4;
    constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * BN;   // two chunk accumulators
    constexpr bool STAGED = BN == 128;       // epilogue stores through shared memory
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
    const GemmArgs& a = p.s;
    // The CTA's work list lives in shared memory: the epilogue warps need their
    // registers for the 128-column running sums.
    __shared__ CtaWork w_s;
    const CtaWork& w = w_s;
    volatile int* abort_flag = &abort_s;

    if (threadIdx.x == 0) {
        w_s = make_work(a, blockIdx.x);
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
            int m0 = 0, n0 = 0, tile = -1;
            Cursor cur;
            cur.seek(w, 0);
            for (; cur.c < w.total; cur.advance(w)) {
                if (cur.tile != tile) {
                    tile = cur.tile;
                    tile_origin(a, tile, BM, BN, m0, n0);
                }
                if (!async::mbar_wait(su32(&empty_bar[stage]), phase ^ 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = su32(&full_bar[stage]);
                const uint32_t base = smem0 + stage * STAGE_BYTES;
                const int k0 = cur.kt * BKT;
                mbar_expect_tx(fb, STAGE_BYTES);
                tma_load_2d(base, &p.tm_ahi, k0, m0, fb);
                tma_load_2d(base + A_BYTES, &p.tm_alo, k0, m0, fb);
                tma_load_2d(base + 2 * A_BYTES, &p.tm_bhi, k0, n0, fb);
                tma_load_2d(base + 2 * A_BYTES + B_BYTES, &p.tm_blo, k0, n0, fb);
                issued[stage] = true;
                issued_phase[stage] = phase;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
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
            Cursor cur;
            cur.seek(w, 0);
            while (ok && cur.c < w.total) {
                // one chunk: k-blocks up to the next multiple of KC_BLOCKS or the end
                // of this CTA's part of the tile
                if (!async::mbar_wait(su32(&tempty_bar[buf]), buf_phase ^ 1u, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                bool first = true, end_chunk = false;
                while (!end_chunk) {
                    if (!async::mbar_wait(su32(&full_bar[stage]), phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = smem0 + stage * STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < BKT / UMMA_K; ++k) {
                        const uint32_t off = k * UMMA_K * 4;
                        const uint64_t ahi = kmajor_desc<BKT>(base + off);
                        const uint64_t alo = kmajor_desc<BKT>(base + A_BYTES + off);
                        const uint64_t bhi = kmajor_desc<BKT>(base + 2 * A_BYTES + off);
                        const uint64_t blo = kmajor_desc<BKT>(base + 2 * A_BYTES + B_BYTES + off);
                        umma_tf32(d_tmem, alo, bhi, idesc, (first && k == 0) ? 0u : 1u);
                        umma_tf32(d_tmem, ahi, blo, idesc, 1u);
                        umma_tf32(d_tmem, ahi, bhi, idesc, 1u);
                    }
                    umma_commit(su32(&empty_bar[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    first = false;
                    end_chunk = (cur.kt + 1 == cur.kt_end) || ((cur.kt + 1) % KC_BLOCKS == 0);
                    cur.advance(w);
                }
                if (!ok) break;
                umma_commit(su32(&tfull_bar[buf]));
                buf ^= 1;
                if (buf == 0) buf_phase ^= 1u;
            }
        }
    } else {
        // ---------------- epilogue: TMEM chunks -> fp32 sums -> C or a partial ----------------
        // Warp w may read TMEM lanes [32 (w % 4), +32) = 32 rows of the tile; the
        // epilogue warps come in groups of four, group g owning columns
        // [128 g, 128 g + 128).
        constexpr int EC = 128;            // accumulator columns per epilogue warp
        const int q = warp & 3;
        const int col0 = EC * ((warp - 2) / 4);
        float* const stg =
            reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES) + (warp - 2) * kStageFloats;
        (void)stg;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        Cursor cur;
        cur.seek(w, 0);
        while (ok && cur.c < w.total) {
            const int tile = cur.tile, kt_begin = cur.kt_begin, kt_end = cur.kt_end;
            int m0, n0;
            tile_origin(a, tile, BM, BN, m0, n0);
            float sum[EC];
#pragma unroll
            for (int i = 0; i < EC; ++i) sum[i] = 0.0f;
            for (;;) {
                const int ce = min(kt_end, (cur.kt / KC_BLOCKS + 1) * KC_BLOCKS);
                if (!async::mbar_wait(su32(&tfull_bar[buf]), buf_phase, abort_flag, a.status)) {
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
                cur.seek(w, cur.c + (ce - cur.kt));
                if (ce == kt_end) break;
            }
            if (!ok) break;
            const bool partial = kt_begin != 0 || kt_end != a.KT;
            float* P = partial ? a.ws_partial + (static_cast<long long>(w.g) * 2 +
                                                 sk_slot(w, tile - w.dp_tiles)) * (BM * BN)
                               : nullptr;
            if constexpr (!STAGED) {
                // Each lane stores its own row (the 256-wide variant has neither the
                // registers nor the shared memory for the staging block).
                const int tr = 32 * q + lane;
#pragma unroll
                for (int u = 0; u < EC / 4; ++u) {
                    const float4 v = make_float4(sum[4 * u], sum[4 * u + 1], sum[4 * u + 2],
                                                 sum[4 * u + 3]);
                    const int tc = col0 + 4 * u;
                    if (partial)
                        __stcg(reinterpret_cast<float4*>(P + tr * BN + tc), v);
                    else if (m0 + tr < a.M)
                        store_c4(a, a.C + static_cast<long long>(m0 + tr) * a.ldc, n0 + tc, v);
                }
            } else {
                // Stores go through a 32 x 32 staging block per warp (16-byte chunks
                // XOR-swizzled by row, so both the row-wise writes and the column-wise
                // reads are conflict-free): each store instruction then covers four
                // whole 128-byte row segments instead of 32 scattered 16-byte pieces.
#pragma unroll
                for (int j = 0; j < EC / 32; ++j) {
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4*>(stg + lane * 32 + ((u ^ (lane & 7)) * 4)) =
                            make_float4(sum[32 * j + 4 * u], sum[32 * j + 4 * u + 1],
                                        sum[32 * j + 4 * u + 2], sum[32 * j + 4 * u + 3]);
                    __syncwarp();
                    const int c4 = lane & 7;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3);            // row in the block
                        const float4 v =
                            *reinterpret_cast<const float4*>(stg + rr * 32 + ((c4 ^ (rr & 7)) * 4));
                        const int tr = 32 * q + rr;                    // row of the tile
                        const int tc = col0 + 32 * j + 4 * c4;         // column of the tile
                        if (partial) {
                            __stcg(reinterpret_cast<float4*>(P + tr * BN + tc), v);
                        } else if (m0 + tr < a.M) {
                            store_c4(a, a.C + static_cast<long long>(m0 + tr) * a.ldc, n0 + tc, v);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // Every store of this CTA is issued: a dependent reduction may start.
    asm volatile("griddepcontrol.launch_dependents;");
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

// Ahi/Alo[i*Kp + k] for i < M, k < Kp (zeros for K <= k < Kp): chunk e of the
// M x Kp/4 float4 chunks is row e / (Kp/4), k = 4 (e % (Kp/4)).  Each chunk is
// read as one float4 when A's row is 16-byte aligned (vec_in) and whole.  hi may
// be null: the GEMM then reads hi straight from A (see below).
__device__ __forceinline__ void split_a_chunk(const float* __restrict__ A, long long lda, int K,
                                              int Kp, int vec_in, long long e,
                                              float* __restrict__ hi, float* __restrict__ lo) {
    const int kp4 = Kp / 4;
    const long long i = e / kp4;
    const int k = 4 * static_cast<int>(e - i * kp4);
    const float* arow = A + i * lda;
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
    const long long o = i * Kp + k;
    if (hi != nullptr) *reinterpret_cast<float4*>(hi + o) = make_float4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<float4*>(lo + o) = make_float4(l[0], l[1], l[2], l[3]);
}

// Bhi/Blo[n*Kp + k] = split(B[k*ldb + n]) for the tile of kTK k by kTN n at
// (k0, n0), through shared memory (row stride kTN + 1: conflict-free transposed
// reads): reads along n and writes along k, both as float4 (reads fall back to
// scalars when B's rows are not 16-byte aligned).  16.6 KB of shared memory, so
// the split kernel keeps full occupancy for the blocks that split A.
constexpr int kTK = 32, kTN = 64;
__device__ __forceinline__ void split_bt_tile(const float* __restrict__ B, long long ldb, int K,
                                              int N, int Kp, int vec_in, int k0, int n0,
                                              float (&th)[kTK][kTN + 1],
                                              float (&tl)[kTK][kTN + 1],
                                              float* __restrict__ hi, float* __restrict__ lo) {
    {
        const int c4 = (threadIdx.x & 15) * 4;   // n within the tile: 16 threads x 4
        const int r0 = threadIdx.x >> 4;         // k within the tile: 16 rows per pass
#pragma unroll
        for (int pass = 0; pass < kTK / 16; ++pass) {
            const int r = r0 + 16 * pass;
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
    }
    __syncthreads();
    {
        const int c4 = (threadIdx.x & 7) * 4;    // k within the tile: 8 threads x 4
        const int r0 = threadIdx.x >> 3;         // n within the tile: 32 rows per pass
#pragma unroll
        for (int pass = 0; pass < kTN / 32; ++pass) {
            const int nr = r0 + 32 * pass;
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
    __syncthreads();
}

// Both splits in one launch: blocks [0, a_blocks) stride over A's float4 chunks,
// the others take the tiles of B in turn.
__global__ void __launch_bounds__(256) split_kernel(
    const float* __restrict__ A, long long lda, int M, const float* __restrict__ B,
    long long ldb, int N, int K, int Kp, int a_vec, int b_vec, int a_blocks,
    float* __restrict__ ahi, float* __restrict__ alo, float* __restrict__ bhi,
    float* __restrict__ blo) {
    if (static_cast<int>(blockIdx.x) < a_blocks) {
        const long long chunks = static_cast<long long>(M) * (Kp / 4);
        for (long long e = blockIdx.x * 256LL + threadIdx.x; e < chunks;
             e += static_cast<long long>(a_blocks) * 256)
            split_a_chunk(A, lda, K, Kp, a_vec, e, ahi, alo);
        return;
    }
    __shared__ float th[kTK][kTN + 1];
    __shared__ float tl[kTK][kTN + 1];
    const int tiles_n = (N + kTN - 1) / kTN;
    const long long tiles = static_cast<long long>(tiles_n) * ((Kp + kTK - 1) / kTK);
    const int b_blocks = static_cast<int>(gridDim.x) - a_blocks;
    for (long long t = static_cast<int>(blockIdx.x) - a_blocks; t < tiles; t += b_blocks) {
        const int tk = static_cast<int>(t / tiles_n);
        const int tn = static_cast<int>(t - static_cast<long long>(tk) * tiles_n);
        split_bt_tile(B, ldb, K, N, Kp, b_vec, tk * kTK, tn * kTN, th, tl, bhi, blo);
    }
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
// Two output-tile widths, each with the k-block depth and ring depth that fill
// about 192 KB of shared memory: 128 columns with 32-deep k-blocks and 3 stages
// (64 KB each), 256 columns with 16-deep k-blocks and 4 stages (48 KB each).
// The pipeline depth matters: 128 columns with 2 stages instead of 3 ran 32 %
// slower, so the 256-wide tile trades k-block depth for stages.  The 128-wide
// tile with 16-deep k-blocks and 6 stages ran 29 % slower than with 32-deep
// blocks and 3: its k-blocks then hold too little MMA work per barrier round.
template <int BN>
struct Variant {
    static constexpr int kBK = BN == 256 ? 16 : 32;
    static constexpr int kStages = BN == 256 ? 4 : 3;
    static constexpr int kThreads = tf32x3_threads(BN);
    static constexpr size_t kSmem =
        static_cast<size_t>(kStages) * (2 * BM * kBK * 4 + 2 * BN * kBK * 4) + 1024 +
        (BN == 128 ? static_cast<size_t>(4) * kStageFloats * 4 : 0);   // + epilogue staging
};

__host__ __device__ constexpr int bk_for(int bn) { return bn == 256 ? 16 : 32; }

// rows x K fp32 matrix with row pitch Kp floats; boxes of bk (K) x box_rows with
// the swizzle the UMMA descriptors expect for bk-float rows.
bool encode_kmajor(CUtensorMap* tm, const float* base, int rows, int K, int Kp, int bk,
                   int box_rows) {
    return encode_fp32_2d(tm, base, rows, K, Kp, bk, box_rows, bk * 4);
}

size_t region_floats(long long rows, int Kp) {
    return align_up_floats(static_cast<size_t>(rows) * Kp);
}

}  // namespace tc

namespace {

int current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

// The schedule of one multiply (one CTA per SM) for tile width bn.
GemmArgs tf32x3_plan(int M, int N, int K, int bn, int sms, int schedule, SchedSizes* z) {
    GemmArgs s{};
    s.M = M;
    s.N = N;
    s.K = K;
    *z = plan_schedule(s, tc::BM, bn, tc::bk_for(bn), sms, 1, schedule);
    return s;
}

struct TcChoice {
    int bn, schedule;
};

// Tile width (128 or 256) and schedule (1: data-parallel only, 0: stream-K on a
// partial last wave or when tiles are fewer than SMs) with the smaller estimated
// time: the k-blocks of the busiest CTA (128-wide: 32 deep, 256-wide: 16 deep), a
// 256-wide 16-deep k-block counting 0.8 128-wide 32-deep ones (measured at 4096^3:
// half the K, twice the columns, the A tile re-read for twice the columns and a
// four-stage ring), plus, when tiles are split, 8 k-blocks for the reduction launch and,
// per 128 columns of split tile, 0.12 (128-wide: staged, coalesced partial
// stores) or 0.55 (256-wide: a row per lane) for writing and re-reading its
// partials (fitted to measured times at 1024^3 .. 8192^3 and the ragged and
// tall shapes).
// SGEMM_TF32X3_BN and SGEMM_TF32X3_SCHEDULE (0 auto, 1 data-parallel, 2
// stream-K whenever possible) override it for tests and tuning.
TcChoice tf32x3_choice(int M, int N, int K, int sms) {
    int force_bn = 0, force_sched = -1;
    if (const char* env = std::getenv("SGEMM_TF32X3_BN")) {
        const int bn = std::atoi(env);
        if (bn == 128 || bn == 256) force_bn = bn;
    }
    if (const char* env = std::getenv("SGEMM_TF32X3_SCHEDULE")) {
        const int v = std::atoi(env);
        if (v >= 0 && v <= 2) force_sched = v;
    }
    TcChoice best{256, 1};
    double best_t = -1.0;
    for (int bn : {256, 128}) {
        if (force_bn && bn != force_bn) continue;
        for (int sched : {1, 0, 2}) {
            if (force_sched >= 0 ? sched != force_sched : sched == 2) continue;
            SchedSizes z;
            const GemmArgs s = tf32x3_plan(M, N, K, bn, sms, sched, &z);
            const long long dp_per = (static_cast<long long>(s.dp_tiles) + s.grid - 1) / s.grid;
            const long long sk_per = (s.sk_iters + s.grid - 1) / s.grid;
            const double split_cost =
                s.sk_tiles > 0 ? 8.0 + (bn == 256 ? 0.55 : 0.12) * s.sk_tiles * (bn / 128) : 0.0;
            const double t =
                static_cast<double>(dp_per * s.KT + sk_per) * (bn == 256 ? 0.8 : 1.0) + split_cost;
            if (best_t < 0.0 || t < best_t) {
                best_t = t;
                best = TcChoice{bn, sched};
            }
        }
    }
    return best;
}

}  // namespace

size_t tf32x3_workspace_bytes(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    const int Kp = (K + 3) / 4 * 4;
    const int sms = current_sms();
    size_t partial = 0;
    if (sms > 0) {
        SchedSizes z;
        const TcChoice c = tf32x3_choice(M, N, K, sms);
        tf32x3_plan(M, N, K, c.bn, sms, c.schedule, &z);
        partial = z.partial_bytes;
    }
    return 4 * (2 * tc::region_floats(M, Kp) + 2 * tc::region_floats(N, Kp)) + partial;
}

namespace {
struct WsLayout {
    float *ahi, *alo, *bhi, *blo, *partial;
};
WsLayout ws_layout(void* ws, int M, int N, int Kp) {
    WsLayout L;
    L.ahi = static_cast<float*>(ws);
    L.alo = L.ahi + tc::region_floats(M, Kp);
    L.bhi = L.alo + tc::region_floats(M, Kp);
    L.blo = L.bhi + tc::region_floats(N, Kp);
    L.partial = L.blo + tc::region_floats(N, Kp);
    return L;
}
}  // namespace

int tf32x3_prepare(int M, int N, int K, const float* A, long long lda, const float* B,
                   long long ldb, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                   bool write_ahi) {
    using namespace tc;
    if (ws == nullptr || ws_bytes < tf32x3_workspace_bytes(M, N, K)) {
        set_last_error_message("tf32x3: workspace too small");
        return SGEMM_ERR_WORKSPACE;
    }
    const int Kp = (K + 3) / 4 * 4;
    const WsLayout L = ws_layout(ws, M, N, Kp);
    const int a_vec = ((reinterpret_cast<uintptr_t>(A) & 15) == 0 && lda % 4 == 0) ? 1 : 0;
    const int b_vec = ((reinterpret_cast<uintptr_t>(B) & 15) == 0 && ldb % 4 == 0) ? 1 : 0;
    // One float4 chunk of A per thread and one 32 x 64 tile of B per block (the
    // kernel strides if the grid would exceed the launch limit): plenty of loads
    // in flight for large operands, and a single launch for small ones.
    const long long a_chunks = static_cast<long long>(M) * (Kp / 4);
    const long long b_tiles = static_cast<long long>((N + kTN - 1) / kTN) * ((Kp + kTK - 1) / kTK);
    const long long cap = 1LL << 30;
    const long long a_blocks = std::min((a_chunks + 255) / 256, cap);
    const long long b_blocks = std::min(b_tiles, cap);
    (void)sms;
    split_kernel<<<static_cast<unsigned>(a_blocks + b_blocks), 256, 0, stream>>>(
        A, lda, M, B, ldb, N, K, Kp, a_vec, b_vec, static_cast<int>(a_blocks),
        write_ahi ? L.ahi : nullptr, L.alo, L.bhi, L.blo);
    if (cudaGetLastError() != cudaSuccess) {
        set_last_error_message("tf32x3: split kernels failed to launch");
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

namespace {

// The shared-memory limit is an attribute of the kernel in each device's context:
// it is raised once per (tile width, device) and forgotten by sgemm_shutdown, so a
// context created after a device reset gets it again.
std::mutex g_attr_mu;
std::vector<int> g_attr_done[2];   // [BN == 256][device]: 0 not yet, 1 done

template <int BN>
int launch_variant(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                   int c_vec, const WsLayout& L, const float* a_hi, long long lda_hi,
                   size_t partial_bytes, int Kp, int sms, int schedule, cudaStream_t stream,
                   int* launches) {
    using namespace tc;
    using V = Variant<BN>;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            set_last_error_message("tf32x3: cudaGetDevice failed");
            return SGEMM_ERR_LAUNCH;
        }
        std::lock_guard<std::mutex> lk(g_attr_mu);
        std::vector<int>& attr_done = g_attr_done[BN == 256 ? 1 : 0];
        if (static_cast<int>(attr_done.size()) <= dev) attr_done.resize(dev + 1, 0);
        if (!attr_done[dev]) {
            if (cudaFuncSetAttribute(tf32x3_kernel<BN, V::kBK, V::kStages>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(V::kSmem)) != cudaSuccess) {
                set_last_error_message("tf32x3: cannot set the kernel's shared-memory size");
                return SGEMM_ERR_LAUNCH;
            }
            attr_done[dev] = 1;
        }
    }
    Params p{};
    // The Ahi operand is A itself when the caller's A can be read by TMA: the
    // tensor core reads an fp32 operand as TF32 by dropping its 13 low mantissa
    // bits, which is exactly hi (measured bit for bit against the split's hi).
    const bool direct = a_hi != nullptr;
    if (!encode_kmajor(&p.tm_ahi, direct ? a_hi : L.ahi, M, K, direct ? lda_hi : Kp, V::kBK,
                       BM) ||
        !encode_kmajor(&p.tm_alo, L.alo, M, K, Kp, V::kBK, BM) ||
        !encode_kmajor(&p.tm_bhi, L.bhi, N, K, Kp, V::kBK, BN) ||
        !encode_kmajor(&p.tm_blo, L.blo, N, K, Kp, V::kBK, BN)) {
        set_last_error_message("tf32x3: cuTensorMapEncodeTiled failed");
        return SGEMM_ERR_LAUNCH;
    }
    SchedSizes z;
    p.s = tf32x3_plan(M, N, K, BN, sms, schedule, &z);
    if (z.partial_bytes > partial_bytes) {
        set_last_error_message("tf32x3: workspace too small for the split tiles");
        return SGEMM_ERR_WORKSPACE;
    }
    p.s.C = C;
    p.s.ldc = ldc;
    p.s.c_vec = c_vec;
    p.s.alpha = alpha;
    p.s.beta = beta;
    p.s.epi = (beta != 0.0f) ? kEpiAlphaBeta : (alpha != 1.0f ? kEpiAlpha : kEpiPlain);
    p.s.ws_partial = L.partial;
    p.s.status = status_word_ptr();
    tf32x3_kernel<BN, V::kBK, V::kStages><<<p.s.grid, V::kThreads, V::kSmem, stream>>>(p);
    *launches = 1;
    if (cudaGetLastError() != cudaSuccess) {
        set_last_error_message("tf32x3: GEMM kernel failed to launch");
        return SGEMM_ERR_LAUNCH;
    }
    if (p.s.sk_tiles > 0) {
        if (launch_sk_reduce(p.s, BM, BN, sms, stream) != cudaSuccess) {
            set_last_error_message("tf32x3: split-tile reduction failed to launch");
            return SGEMM_ERR_LAUNCH;
        }
        *launches = 2;
    }
    return SGEMM_OK;
}

}  // namespace

void forget_tf32x3_attributes() {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (auto& v : g_attr_done) v.clear();
}

int tf32x3_tile_width(int M, int N, int K, int sms) {
    return tf32x3_choice(M, N, K, sms).bn;
}

int tf32x3_query(int M, int N, int K, int sms, sgemm_config* out) {
    const TcChoice c = tf32x3_choice(M, N, K, sms);
    const int bn = c.bn;
    SchedSizes z;
    const GemmArgs s = tf32x3_plan(M, N, K, bn, sms, c.schedule, &z);
    const bool wide = bn == 256;
    out->bm = tc::BM;
    out->bn = bn;
    out->bk = tc::bk_for(bn);
    out->wm = 32;
    out->wn = 128;
    out->tm = 1;
    out->tn = 128;
    out->stages = wide ? tc::Variant<256>::kStages : tc::Variant<128>::kStages;
    out->threads = tc::tf32x3_threads(bn);
    out->smem_bytes = static_cast<int>(wide ? tc::Variant<256>::kSmem : tc::Variant<128>::kSmem);
    out->split_k = z.split;
    out->kernel_id = -1;
    out->vec = 4;
    out->grid = s.grid;
    out->tiles = s.tiles_m * s.tiles_n;
    out->sk_tiles = s.sk_tiles;
    out->ctas_per_sm = 1;
    out->fma2 = 0;
    out->packed = 0;
    out->sk_gap = s.sk_gap;
    return SGEMM_OK;
}

int tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                    int c_vec, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                    int* launches, const float* a_hi, long long lda_hi) {
    *launches = 0;
    const size_t need = tf32x3_workspace_bytes(M, N, K);
    if (ws == nullptr || ws_bytes < need) {
        set_last_error_message("tf32x3: workspace too small");
        return SGEMM_ERR_WORKSPACE;
    }
    const int Kp = (K + 3) / 4 * 4;
    const WsLayout L = ws_layout(ws, M, N, Kp);
    const size_t partial_bytes =
        ws_bytes - static_cast<size_t>(reinterpret_cast<char*>(L.partial) -
                                       static_cast<char*>(ws));
    const TcChoice c = tf32x3_choice(M, N, K, sms);
    if (c.bn == 256)
        return launch_variant<256>(M, N, K, alpha, beta, C, ldc, c_vec, L, a_hi, lda_hi,
                                   partial_bytes, Kp, sms, c.schedule, stream, launches);
    return launch_variant<128>(M, N, K, alpha, beta, C, ldc, c_vec, L, a_hi, lda_hi,
                               partial_bytes, Kp, sms, c.schedule, stream, launches);
}

}  // namespace sgemm
