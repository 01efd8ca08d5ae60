// FP32 SGEMM on the CUDA cores of sm_103a: persistent, multistage cp.async
// pipeline, register outer-product micro-kernel, stream-K tail balancing.
//
// The hierarchy is the one the source pages describe ("누산 개념을
// Grid-Block-Warp-Thread 계층에 끼워넣기", §2 (1)-(4); "Register/Shared Memory
// Tiling", 동작 원리 and 아웃터 프로덕트 GEMM):
//   * a CTA computes BM x BN tiles of C,
//   * a warp owns a WM x WN warp tile inside the CTA tile,
//   * a thread owns a TM x TN register tile acc[TM][TN],
//   * the K range is walked in BK-deep slices staged in shared memory, and
//     every k of a slice applies the rank-1 update acc[i][j] += a[i] * b[j]
//     ("기존 작성한 GE_v2 의 regemm 타일드 커널의 1:1 매핑, gemm_tiled_test 작성",
//     §5: one fmaf per accumulator per k).
//
// What is different from the pages' kernels, and why (GB300 first):
//   * Loads are cp.async (16-byte .cg when rows are 16-byte aligned, 4-byte .ca
//     otherwise) into a STAGES-deep ring of shared-memory slices instead of the
//     pages' synchronous single / double buffer ("Register/Shared Memory
//     Tiling", 더블 버퍼링 구현), so global latency overlaps several slices of math.
//   * Out-of-range elements are zero-filled by the copy itself (src-size 0 or a
//     short src-size), which is the pages' "boundary check then 0-padding"
//     (GE_v2 page, §3) without a branch around the copy.
//   * The A slice keeps its global row-major layout with a 4-float row pad; a
//     thread reads AK consecutive k of one row per LDS, and the odd row stride
//     in 16-byte units puts the LR rows a warp reads in distinct banks.  The B
//     slice is unpadded; each LDS.128 of a warp touches LC consecutive 16-byte
//     chunks of one row.  (The pages' `+PADK/+PADN` padding, GE_v2 page §2.)
//   * The copies of the next slice of an interior tile go out in parts spread
//     over the current slice's k-steps (SPREAD), not in one burst before it: data
//     landing in shared memory all at once holds up the fragment loads.
//   * The grid is persistent (SM count x resident CTAs).  Each CTA walks a flat
//     list of k-slices that may cross tile boundaries, so the copy pipeline
//     never drains between tiles.  Whole waves of tiles are data-parallel; the
//     last partial wave is shared out by k-slices over all CTAs (stream-K).  Each
//     CTA writes its partial tiles to a workspace and a second, bandwidth-bound
//     kernel (sgemm_reduce.cu) sums every split tile's partials over all SMs in
//     a fixed order, so results are identical from run to run.
//   * Problems of less than one resident wave may instead split every tile over
//     a thread-block cluster whose CTAs sum their partial tiles in distributed
//     shared memory, in k order, inside the same launch (cluster_sum_store).
#pragma once

#include <stdint.h>

#include "sgemm_epilogue.cuh"
#include "sgemm_args.h"
#include "sgemm_sched.cuh"

namespace sgemm {

// ----------------------------------------------------------------------------
// PTX helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
                 "l"(__cvta_generic_to_global(src)), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst),
                 "l"(__cvta_generic_to_global(src)), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Thread-block cluster primitives (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; shared-memory writes made
// before the arrive are visible to the whole cluster after the wait.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work between them.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the shared::cluster window of the same shared-memory location in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_address, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_address), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t address) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(address)
                 : "memory");
    return v;
}

// d += x * y elementwise on packed pairs (low 32 bits = column j, high = column
// j+1); one multiplicand is two adjacent B values, the other one A value in both
// halves.  The product is commutative; the operand order is a scheduling choice.
__device__ __forceinline__ void ffma2(unsigned long long& d, unsigned long long x,
                                      unsigned long long y) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(x), "l"(y));
}

// d += {a, a} * b: the A value broadcast into both halves inside the same asm.
__device__ __forceinline__ void ffma2_bcast(unsigned long long& d, float a,
                                            unsigned long long b) {
    asm("{\n\t.reg .b64 ta;\n\t"
        "mov.b64 ta, {%1, %1};\n\t"
        "fma.rn.f32x2 %0, ta, %2, %0;\n\t}"
        : "+l"(d)
        : "f"(a), "l"(b));
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float lo_f(unsigned long long x) {
    return __uint_as_float(static_cast<uint32_t>(x));
}
__device__ __forceinline__ float hi_f(unsigned long long x) {
    return __uint_as_float(static_cast<uint32_t>(x >> 32));
}

// ----------------------------------------------------------------------------
// Register accumulators: plain fp32, or packed pairs for fma.rn.f32x2
// ----------------------------------------------------------------------------
// BOUTER (packed form only): true = one B pair against every A value in turn,
// false = one A value against every B pair.
template <int TM, int TN, bool FMA2, bool BOUTER = true>
struct Acc;

template <int TM, int TN, bool BOUTER>
struct Acc<TM, TN, false, BOUTER> {
    float v[TM][TN];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) v[i][j] = 0.0f;
    }
    // b holds TN values of one k (TN/4 float4 chunks).
    __device__ __forceinline__ void rank1(const float (&a)[TM], const float4 (&b)[TN / 4]) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j4 = 0; j4 < TN / 4; ++j4) {
                v[i][4 * j4 + 0] = fmaf(a[i], b[j4].x, v[i][4 * j4 + 0]);
                v[i][4 * j4 + 1] = fmaf(a[i], b[j4].y, v[i][4 * j4 + 1]);
                v[i][4 * j4 + 2] = fmaf(a[i], b[j4].z, v[i][4 * j4 + 2]);
                v[i][4 * j4 + 3] = fmaf(a[i], b[j4].w, v[i][4 * j4 + 3]);
            }
    }
    __device__ __forceinline__ float4 chunk(int i, int j4) const {
        return make_float4(v[i][4 * j4], v[i][4 * j4 + 1], v[i][4 * j4 + 2], v[i][4 * j4 + 3]);
    }
};

template <int TM, int TN, bool BOUTER>
struct Acc<TM, TN, true, BOUTER> {
    unsigned long long v[TM][TN / 2];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN / 2; ++j) v[i][j] = 0ull;
    }
    // B outer with B as the first multiplicand measured 1-3 % faster on the 8x16
    // tile of the cp.async kernels; it keeps all TM broadcast pairs live, which
    // the TMA kernel (A fragments for two k at once) cannot afford, so that one
    // takes A outer.  The rows run down for even column pairs and back up for odd
    // ones, so the FFMA2s on either side of each turn share their A pair: 1.9 %
    // faster at 4096^3 and 4 % at 1024^3 than restarting every column pair at row 0.
    __device__ __forceinline__ void rank1(const float (&a)[TM], const float4 (&b)[TN / 4]) {
        unsigned long long bp[TN / 2];
#pragma unroll
        for (int j4 = 0; j4 < TN / 4; ++j4) {
            bp[2 * j4] = pack2(b[j4].x, b[j4].y);
            bp[2 * j4 + 1] = pack2(b[j4].z, b[j4].w);
        }
        if constexpr (BOUTER) {
            unsigned long long ap[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i) ap[i] = pack2(a[i], a[i]);
#pragma unroll
            for (int j = 0; j < TN / 2; ++j)
#pragma unroll
                for (int ii = 0; ii < TM; ++ii) {
                    const int i = (j & 1) ? TM - 1 - ii : ii;
                    ffma2(v[i][j], bp[j], ap[i]);
                }
        } else {
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN / 2; ++j) ffma2_bcast(v[i][j], a[i], bp[j]);
        }
    }
    __device__ __forceinline__ float4 chunk(int i, int j4) const {
        return make_float4(lo_f(v[i][2 * j4]), hi_f(v[i][2 * j4]), lo_f(v[i][2 * j4 + 1]),
                           hi_f(v[i][2 * j4 + 1]));
    }
};

// ----------------------------------------------------------------------------
// The kernel
// ----------------------------------------------------------------------------
template <int BM_, int BN_, int BK_, int TM_, int TN_, int LR_, int WARPS_M_, int WARPS_N_,
          int STAGES_, int VEC_, int AK_, bool FMA2_, int MINB_, bool PIPE_ = false,
          int KU_ = 0, int SPREAD_ = 0, int SPREAD_FRAC_ = 1>
struct FfmaCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, TM = TM_, TN = TN_;
    static constexpr int LR = LR_, LC = 32 / LR_;
    static constexpr int WM = TM * LR, WN = TN * LC;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int NT = 32 * WARPS_M * WARPS_N;
    static constexpr int STAGES = STAGES_, VEC = VEC_, AK = AK_;
    static constexpr bool FMA2 = FMA2_;
    static constexpr int MINB = MINB_;
    // PIPE: load the next k's fragments before the current k's FMAs (register
    // double buffering of A and B fragments inside a slice).
    static constexpr bool PIPE = PIPE_;
    // KU: AK-deep steps per copy of the unrolled slice loop (0: the whole slice).
    static constexpr int KU = KU_ > 0 ? KU_ : BK_ / AK_;
    // SPREAD > 0: the refill of the next ring slot is cut into up to SPREAD parts
    // issued at evenly spaced AK-steps of the first loop body of compute_slice,
    // instead of one burst before it (see compute_slice).
    static constexpr int SPREAD = SPREAD_;
    // The parts go into the first 1 / SPREAD_FRAC of the slice's k-steps.
    static constexpr int SPREAD_FRAC = SPREAD_FRAC_;
    // A slice: [BM][BK + PADA] (row stride odd in 16-byte units); B slice: [BK][BN].
    static constexpr int PADA = ((BK / 4) % 2 == 0) ? 4 : 0;
    static constexpr int LDAS = BK + PADA;
    static constexpr int LDBS = BN;
    static constexpr int A_STAGE = BM * LDAS;
    static constexpr int B_STAGE = BK * LDBS;
    // Cluster split: the CTA's partial tile, rows padded by 8 floats so the float4
    // writes of a quarter-warp (4 rows x 2 adjacent chunks) hit distinct banks.
    static constexpr int LDP = BN + 8;
    static constexpr int PART_BYTES = BM * LDP * 4;
    static constexpr int PIPE_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int SMEM_BYTES = PIPE_BYTES > PART_BYTES ? PIPE_BYTES : PART_BYTES;

    static_assert(BM == WM * WARPS_M, "BM must equal WM * WARPS_M");
    static_assert(BN == WN * WARPS_N, "BN must equal WN * WARPS_N");
    static_assert(32 % LR == 0, "LR must divide 32");
    static_assert(TN % 4 == 0, "TN must be a multiple of 4");
    static_assert(BK % 4 == 0 && BK % AK == 0, "BK must be a multiple of 4 and of AK");
    static_assert(AK == 1 || AK == 2 || AK == 4, "AK is 1, 2 or 4");
    static_assert(STAGES >= 2, "at least two stages");
};

// Part p of P of one slice's copies: each thread's copy loops are cut into P
// contiguous ranges of iterations (P = 1, p = 0: the whole slice).
template <class Cfg, int P = 1, int p = 0>
__device__ __forceinline__ void load_slice(const GemmArgs& a, float* sA, float* sB, int m0,
                                           int n0, int k0, int tid) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, NT = Cfg::NT;
    constexpr int LDAS = Cfg::LDAS, LDBS = Cfg::LDBS;
    const int rows_left = a.M - m0;   // valid rows of this A tile: r < rows_left
    const int k_left = a.K - k0;      // valid k of this slice:      c < k_left
    const int cols_left = a.N - n0;   // valid columns of this B tile
    if constexpr (Cfg::VEC == 4) {
        // A: BM rows x BK/4 chunks of 16 bytes.
        constexpr int CPR = BK / 4;
        constexpr int CHUNKS = BM * CPR;
        constexpr int JA = (CHUNKS + NT - 1) / NT;
#pragma unroll
        for (int j = JA * p / P; j < JA * (p + 1) / P; ++j) {
            const int e = j * NT + tid;
            if (CHUNKS % NT == 0 || e < CHUNKS) {
                const int r = e / CPR, c = (e % CPR) * 4;
                const bool ok = (r < rows_left) && (c < k_left);
                const int bytes = ok ? min(16, (k_left - c) * 4) : 0;
                const float* src = ok ? a.A + (m0 + r) * a.lda + (k0 + c) : a.A;
                cp_async16(smem_addr(sA + r * LDAS + c), src, bytes);
            }
        }
        // B: BK rows x BN/4 chunks.
        constexpr int CPRB = BN / 4;
        constexpr int CHUNKSB = BK * CPRB;
        constexpr int JB = (CHUNKSB + NT - 1) / NT;
#pragma unroll
        for (int j = JB * p / P; j < JB * (p + 1) / P; ++j) {
            const int e = j * NT + tid;
            if (CHUNKSB % NT == 0 || e < CHUNKSB) {
                const int r = e / CPRB, c = (e % CPRB) * 4;
                const bool ok = (r < k_left) && (c < cols_left);
                const int bytes = ok ? min(16, (cols_left - c) * 4) : 0;
                const float* src = ok ? a.B + (k0 + r) * a.ldb + (n0 + c) : a.B;
                cp_async16(smem_addr(sB + r * LDBS + c), src, bytes);
            }
        }
    } else {
        constexpr int ELEMS = BM * BK;
        constexpr int JA = (ELEMS + NT - 1) / NT;
#pragma unroll
        for (int j = JA * p / P; j < JA * (p + 1) / P; ++j) {
            const int e = j * NT + tid;
            if (ELEMS % NT == 0 || e < ELEMS) {
                const int r = e / BK, c = e % BK;
                const bool ok = (r < rows_left) && (c < k_left);
                const float* src = ok ? a.A + (m0 + r) * a.lda + (k0 + c) : a.A;
                cp_async4(smem_addr(sA + r * LDAS + c), src, ok ? 4 : 0);
            }
        }
        constexpr int ELEMSB = BK * BN;
        constexpr int JB = (ELEMSB + NT - 1) / NT;
#pragma unroll
        for (int j = JB * p / P; j < JB * (p + 1) / P; ++j) {
            const int e = j * NT + tid;
            if (ELEMSB % NT == 0 || e < ELEMSB) {
                const int r = e / BN, c = e % BN;
                const bool ok = (r < k_left) && (c < cols_left);
                const float* src = ok ? a.B + (k0 + r) * a.ldb + (n0 + c) : a.B;
                cp_async4(smem_addr(sB + r * LDBS + c), src, ok ? 4 : 0);
            }
        }
    }
}

// One BK-deep slice of rank-1 updates from shared memory into the registers.
// Fragments of one slice: A as AK consecutive k of each of the thread's TM rows
// (one 16- or 8-byte load per row), B as TN values of one k.
template <class Cfg>
__device__ __forceinline__ void load_a_frag(const float* sA, int a_row0, int kq,
                                            float (&av)[Cfg::TM][Cfg::AK]) {
    constexpr int TM = Cfg::TM, AK = Cfg::AK, LR = Cfg::LR, LDAS = Cfg::LDAS;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const float* p = sA + (a_row0 + i * LR) * LDAS + kq;
        if constexpr (AK == 4) {
            const float4 t = *reinterpret_cast<const float4*>(p);
            av[i][0] = t.x; av[i][1] = t.y; av[i][2] = t.z; av[i][3] = t.w;
        } else if constexpr (AK == 2) {
            const float2 t = *reinterpret_cast<const float2*>(p);
            av[i][0] = t.x; av[i][1] = t.y;
        } else {
            av[i][0] = *p;
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void load_b_frag(const float* sB, int b_col0, int k,
                                            float4 (&b)[Cfg::TN / 4]) {
#pragma unroll
    for (int j4 = 0; j4 < Cfg::TN / 4; ++j4)
        b[j4] = *reinterpret_cast<const float4*>(sB + k * Cfg::LDBS + b_col0 + j4 * Cfg::LC * 4);
}

// Where the copies of the next slice go while this one is computed.
struct Refill {
    uint32_t sa, sb;     // shared-memory addresses of this thread's first A and B chunks
    const float* ga;     // this thread's first A source of the slice
    const float* gb;     // this thread's first B source
    bool on;             // a slice is to be loaded, spread over this one's compute
};

// Interior slices (every element inside A and B, 16-byte rows): part p of P of
// this thread's copies, with no bounds checks.  Thread t copies chunk t % CPR of
// rows t / CPR + j * RS; part p takes j in [p * JA / P, (p + 1) * JA / P).
template <class Cfg>
struct InteriorCopy {
    static constexpr int CPR = Cfg::BK / 4, RS = Cfg::NT / CPR, JA = Cfg::BM / RS;
    static constexpr int CPRB = Cfg::BN / 4, RSB = Cfg::NT / CPRB, JB = Cfg::BK / RSB;
    static constexpr bool OK = Cfg::VEC == 4 && Cfg::NT % CPR == 0 && Cfg::BM % RS == 0 &&
                               Cfg::NT % CPRB == 0 && Cfg::BK % RSB == 0;
};

template <class Cfg, int P>
__device__ __forceinline__ void refill_part(const GemmArgs& a, const Refill& rf, int p) {
    using IC = InteriorCopy<Cfg>;
    // ceil(J / P) copies per part; the last parts of a loop shorter than P copy less.
    constexpr int NA = (IC::JA + P - 1) / P, NB = (IC::JB + P - 1) / P;
    const long long lda = a.lda, ldb = a.ldb;
    const float* ga = rf.ga + static_cast<long long>(p * NA * IC::RS) * lda;
    const uint32_t sa = rf.sa + static_cast<uint32_t>(p * NA * IC::RS * Cfg::LDAS * 4);
#pragma unroll
    for (int j = 0; j < NA; ++j)
        if (IC::JA % P == 0 || p * NA + j < IC::JA)
            cp_async16(sa + j * IC::RS * Cfg::LDAS * 4, ga + j * IC::RS * lda, 16);
    const float* gb = rf.gb + static_cast<long long>(p * NB * IC::RSB) * ldb;
    const uint32_t sb = rf.sb + static_cast<uint32_t>(p * NB * IC::RSB * Cfg::LDBS * 4);
#pragma unroll
    for (int j = 0; j < NB; ++j)
        if (IC::JB % P == 0 || p * NB + j < IC::JB)
            cp_async16(sb + j * IC::RSB * Cfg::LDBS * 4, gb + j * IC::RSB * ldb, 16);
}

// Shared-memory copies landing in one burst at the start of a slice delay the
// fragment loads behind them: measured on GB300, the 256 x 128 x 64 micro-kernel
// on resident shared memory keeps the FMA pipe 87 % busy with its per-slice
// barrier, 80 % when the next slice's cp.async copies (L2 hits) are issued
// before the slice and 86 % when they are issued in 8 parts over its first half.
// With SPREAD = P > 0 an interior refill is issued in P parts at evenly spaced
// AK-steps of the slice (P / H of them in each of the H loop bodies).
template <class Cfg, class AccT>
__device__ __forceinline__ void compute_slice(const float* sA, const float* sB, int a_row0,
                                              int b_col0, AccT& acc, const GemmArgs& a,
                                              const Refill& rf) {
    constexpr int BK = Cfg::BK, TM = Cfg::TM, TN = Cfg::TN, AK = Cfg::AK;
    constexpr int STEPS = BK / AK / Cfg::SPREAD_FRAC;   // k-steps the parts spread over
    constexpr int P = Cfg::SPREAD;
    static_assert(P == 0 || (STEPS % P == 0), "parts at evenly spaced steps");
    constexpr int SPAN = P > 0 ? STEPS / P : 1;   // AK-steps between two parts
    if constexpr (Cfg::PIPE) {
        // Two fragment sets: the loads for the next step are issued before the
        // current step's FMAs, so shared-memory latency hides behind them.
        float av[2][TM][AK];
        float4 b[2][TN / 4];
        load_a_frag<Cfg>(sA, a_row0, 0, av[0]);
        load_b_frag<Cfg>(sB, b_col0, 0, b[0]);
#pragma unroll
        for (int kq = 0; kq < BK; kq += AK) {
            if constexpr (P > 0) {
                if ((kq / AK) % SPAN == 0 && (kq / AK) / SPAN < P && rf.on)
                    refill_part<Cfg, P>(a, rf, (kq / AK) / SPAN);
            }
            const int ab = (kq / AK) & 1;
            if (kq + AK < BK) load_a_frag<Cfg>(sA, a_row0, kq + AK, av[ab ^ 1]);
#pragma unroll
            for (int kk = 0; kk < AK; ++kk) {
                const int k = kq + kk, bb = k & 1;
                if (k + 1 < BK) load_b_frag<Cfg>(sB, b_col0, k + 1, b[bb ^ 1]);
                float ak[TM];
#pragma unroll
                for (int i = 0; i < TM; ++i) ak[i] = av[ab][i][kk];
                acc.rank1(ak, b[bb]);
            }
        }
    } else {
        // Loop bodies of KU AK-steps.
        constexpr int H = BK / (Cfg::KU * AK);
        static_assert(BK % (Cfg::KU * AK) == 0, "KU steps divide the slice");
        static_assert(P == 0 || Cfg::KU % SPAN == 0, "parts at the same steps of every body");
#pragma unroll 1
        for (int h = 0; h < H; ++h) {
#pragma unroll
            for (int s = 0; s < Cfg::KU; ++s) {
                if constexpr (P > 0) {
                    const int part = h * (Cfg::KU / SPAN) + s / SPAN;
                    if (s % SPAN == 0 && (Cfg::SPREAD_FRAC == 1 || part < P) && rf.on)
                        refill_part<Cfg, P>(a, rf, part);
                }
                const int kq = (h * Cfg::KU + s) * AK;
                float av[TM][AK];
                load_a_frag<Cfg>(sA, a_row0, kq, av);
#pragma unroll
                for (int kk = 0; kk < AK; ++kk) {
                    float4 b[TN / 4];
                    load_b_frag<Cfg>(sB, b_col0, kq + kk, b);
                    float ak[TM];
#pragma unroll
                    for (int i = 0; i < TM; ++i) ak[i] = av[i][kk];
                    acc.rank1(ak, b);
                }
            }
        }
    }
}

template <class Cfg, class AccT>
__device__ __forceinline__ void store_tile(const GemmArgs& a, const AccT& acc, int m0, int n0,
                                           int a_row0, int b_col0) {
    constexpr int TM = Cfg::TM, TN = Cfg::TN, LR = Cfg::LR, LC = Cfg::LC;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + a_row0 + i * LR;
        if (gm >= a.M) continue;
        float* crow = a.C + gm * a.ldc;
#pragma unroll
        for (int j4 = 0; j4 < TN / 4; ++j4)
            store_c4(a, crow, n0 + b_col0 + j4 * LC * 4, acc.chunk(i, j4));
    }
}

// Split tile: write this CTA's partial sum of the tile (tile-local row-major
// BM x BN floats) to its workspace slot.  sk_reduce_kernel adds the partials up.
template <class Cfg, class AccT>
__device__ __forceinline__ void store_partial(const GemmArgs& a, const CtaWork& w,
                                              const Cursor& cur, const AccT& acc, int a_row0,
                                              int b_col0) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, TM = Cfg::TM, TN = Cfg::TN;
    constexpr int LR = Cfg::LR, LC = Cfg::LC;
    const int t = cur.tile - w.dp_tiles;           // index among split tiles
    float* P = a.ws_partial + (static_cast<long long>(w.g) * 2 + sk_slot(w, t)) * (BM * BN);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j4 = 0; j4 < TN / 4; ++j4)
            __stcg(reinterpret_cast<float4*>(P + (a_row0 + i * LR) * BN + b_col0 + j4 * LC * 4),
                   acc.chunk(i, j4));
}

// Cluster split: rank r of the S CTAs sharing a tile sums rows
// [r*BM/S, (r+1)*BM/S) of the S partial tiles, held in the CTAs' shared memory,
// in rank order (rank q computed the q-th contiguous piece of K, so this is
// increasing k, as in the stream-K reduction), and stores them to C.  Each
// thread first issues all the distributed-shared-memory loads of U float4 of
// the band, then adds and stores them.
template <class Cfg, int S>
__device__ __forceinline__ void cluster_band_sum(const GemmArgs& a, const float* part, int tid) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, NT = Cfg::NT, LDP = Cfg::LDP;
    static_assert(BM % S == 0, "the cluster size divides the tile height");
    constexpr int ROWS = BM / S;
    constexpr int CPR = BN / 4;                      // float4 per row
    constexpr int V4 = ROWS * CPR;                   // float4 in this CTA's band
    constexpr int PER = (V4 + NT - 1) / NT;          // float4 per thread
    constexpr int U0 = (32 / S) < 1 ? 1 : 32 / S;    // at most 32 loads in flight
    constexpr int U = PER < U0 ? PER : U0;
    const uint32_t rank = cluster_ctarank();
    const int tile = blockIdx.x / S;
    int m0, n0;
    tile_origin(a, a.dp_tiles + tile, BM, BN, m0, n0);
    const uint32_t base = smem_addr(part);
    uint32_t peer[S];
#pragma unroll
    for (int q = 0; q < S; ++q) peer[q] = map_to_rank(base, static_cast<uint32_t>(q));
    const int row0 = static_cast<int>(rank) * ROWS;
    for (int e0 = 0; e0 < PER; e0 += U) {
        float4 v[U][S];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = (e0 + u) * NT + tid;
            if ((V4 % NT == 0 || e < V4) && e0 + u < PER) {
                const int rr = row0 + e / CPR, cc = (e % CPR) * 4;
                const uint32_t off = static_cast<uint32_t>((rr * LDP + cc) * 4);
#pragma unroll
                for (int q = 0; q < S; ++q) v[u][q] = ld_cluster_f4(peer[q] + off);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = (e0 + u) * NT + tid;
            if ((V4 % NT == 0 || e < V4) && e0 + u < PER) {
                float4 t = v[u][0];
#pragma unroll
                for (int q = 1; q < S; ++q) {
                    t.x += v[u][q].x;
                    t.y += v[u][q].y;
                    t.z += v[u][q].z;
                    t.w += v[u][q].w;
                }
                v[u][0] = t;
            }
        }
        // After the last batch every value this thread reads from its peers is
        // in registers: tell the cluster so (the matching wait is at the end).
        if (e0 + U >= PER) cluster_arrive();
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = (e0 + u) * NT + tid;
            if ((V4 % NT == 0 || e < V4) && e0 + u < PER) {
                const int gm = m0 + row0 + e / CPR, gn = n0 + (e % CPR) * 4;
                if (gm < a.M && gn < a.N) store_c4(a, a.C + gm * a.ldc, gn, v[u][0]);
            }
        }
    }
}

// The end of a cluster-split CTA: its partial tile goes to its own shared memory
// (the pipeline slices are free by now), the cluster synchronises, each CTA sums
// its band of rows over the cluster, and a second cluster barrier (arrive once
// the peers' values are read, wait before exit) keeps every CTA's shared memory
// alive until all peers have read it.  Every thread of every CTA of the cluster
// reaches both barriers: cluster_band_sum arrives exactly once per thread (its
// batch loop runs at least once, PER >= 1), and S is 2, 4 or 8.
template <class Cfg, class AccT>
__device__ __forceinline__ void cluster_sum_store(const GemmArgs& a, const AccT& acc,
                                                  float* part, int a_row0, int b_col0,
                                                  int tid) {
    constexpr int TM = Cfg::TM, TN = Cfg::TN, LR = Cfg::LR, LC = Cfg::LC, LDP = Cfg::LDP;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j4 = 0; j4 < TN / 4; ++j4)
            *reinterpret_cast<float4*>(part + (a_row0 + i * LR) * LDP + b_col0 + j4 * LC * 4) =
                acc.chunk(i, j4);
    cluster_sync();
    switch (a.cl_split) {
        case 2: cluster_band_sum<Cfg, 2>(a, part, tid); break;
        case 4: cluster_band_sum<Cfg, 4>(a, part, tid); break;
        case 8: cluster_band_sum<Cfg, 8>(a, part, tid); break;
        default: cluster_arrive(); break;
    }
    cluster_wait();
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MINB) sgemm_ffma_kernel(const GemmArgs a) {
    extern __shared__ __align__(16) float smem[];
    constexpr int STAGES = Cfg::STAGES, BK = Cfg::BK;
    using AccT = Acc<Cfg::TM, Cfg::TN, Cfg::FMA2>;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp / Cfg::WARPS_N, warp_n = warp % Cfg::WARPS_N;
    // Lane -> (lr, lc).  Each quarter-warp (8 lanes, the unit a 16-byte shared
    // load is served in) holds LRQ lane-rows x LCQ lane-columns, so one LDS.128
    // of a quarter-warp touches at most LRQ distinct A rows or LCQ adjacent B
    // chunks, in disjoint banks, and is served at the broadcast rate.
    constexpr int LRQ = Cfg::LR < 8 ? Cfg::LR : 8;
    constexpr int LCQ = 8 / LRQ;
    const int q = lane >> 3, li = lane & 7;
    const int lr = (q % (Cfg::LR / LRQ)) * LRQ + li % LRQ;
    const int lc = (q / (Cfg::LR / LRQ)) * LCQ + li / LRQ;
    // First A row / B column of this thread inside the CTA tile.  Rows are
    // interleaved by LR, column chunks by LC*4.
    const int a_row0 = warp_m * Cfg::WM + lr;
    const int b_col0 = warp_n * Cfg::WN + lc * 4;

    // A cluster-split CTA always goes on to the cluster barriers at the end.
    const bool cl = a.cl_split > 1;
    const CtaWork w = cl ? make_cluster_work(a, blockIdx.x) : make_work(a, blockIdx.x);
    if (w.total <= 0 && !cl) return;

    float* const sA0 = smem;
    float* const sB0 = smem + STAGES * Cfg::A_STAGE;

    Cursor ld;
    if (cl) {
        const int t = static_cast<int>(blockIdx.x) >> (__ffs(a.cl_split) - 1);
        const long long tb = static_cast<long long>(t) * w.KT;
        ld.set_piece(t, static_cast<int>(w.u0 - tb), static_cast<int>(w.u1 - tb));
    } else {
        ld.seek(w, 0);
    }
    Cursor cp = ld;

    // Launched as a programmatic dependent of the stream's previous kernel: the
    // set-up above overlaps that kernel's tail, and nothing in global memory is
    // read or written before it has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Prologue: fill STAGES-1 slices.
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (ld.c < w.total) {
            int m0, n0;
            tile_origin(a, ld.tile, Cfg::BM, Cfg::BN, m0, n0);
            load_slice<Cfg>(a, sA0 + s * Cfg::A_STAGE, sB0 + s * Cfg::B_STAGE, m0, n0,
                            ld.kt * BK, tid);
            ld.advance(w);
        }
        cp_async_commit();
    }

    AccT acc;
    acc.zero();
    int stage = 0;
    int m0c, n0c;
    tile_origin(a, cp.tile, Cfg::BM, Cfg::BN, m0c, n0c);

    for (long long c = 0; c < w.total; ++c) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        // Refill the slot computed in the previous iteration: in one burst here, or
        // spread over the first loop body of this slice's compute (SPREAD).
        Refill rf;
        rf.on = false;
        if (ld.c < w.total) {
            const int ls = (stage + STAGES - 1) % STAGES;
            float* const la = sA0 + ls * Cfg::A_STAGE;
            float* const lb = sB0 + ls * Cfg::B_STAGE;
            int m0, n0;
            tile_origin(a, ld.tile, Cfg::BM, Cfg::BN, m0, n0);
            const int k0 = ld.kt * BK;
            ld.advance(w);
            if constexpr (Cfg::SPREAD > 0) {
                using IC = InteriorCopy<Cfg>;
                static_assert(IC::OK, "spread refills need the 16-byte interior copy layout");
                rf.on = m0 + Cfg::BM <= a.M && n0 + Cfg::BN <= a.N && k0 + BK <= a.K;
                if (rf.on) {
                    const int ra = tid / IC::CPR, ca = (tid % IC::CPR) * 4;
                    const int rb = tid / IC::CPRB, cb = (tid % IC::CPRB) * 4;
                    rf.sa = smem_addr(la + ra * Cfg::LDAS + ca);
                    rf.sb = smem_addr(lb + rb * Cfg::LDBS + cb);
                    rf.ga = a.A + static_cast<long long>(m0 + ra) * a.lda + (k0 + ca);
                    rf.gb = a.B + static_cast<long long>(k0 + rb) * a.ldb + (n0 + cb);
                }
            }
            // Edge slices (and SPREAD = 0): the whole slice now, bounds checked.
            if (!rf.on) load_slice<Cfg>(a, la, lb, m0, n0, k0, tid);
        }

        compute_slice<Cfg>(sA0 + stage * Cfg::A_STAGE, sB0 + stage * Cfg::B_STAGE, a_row0,
                           b_col0, acc, a, rf);
        cp_async_commit();
        stage = (stage + 1 == STAGES) ? 0 : stage + 1;

        if (cp.kt + 1 == cp.kt_end) {
            // A cluster-split CTA holds one piece of one tile: its sum stays in
            // the registers for the cluster sum after the loop.
            if (!cl) {
                if (cp.kt_begin == 0 && cp.kt_end == w.KT)
                    store_tile<Cfg>(a, acc, m0c, n0c, a_row0, b_col0);
                else
                    store_partial<Cfg>(a, w, cp, acc, a_row0, b_col0);
                acc.zero();
            }
            cp.advance(w);
            if (cp.c < w.total) tile_origin(a, cp.tile, Cfg::BM, Cfg::BN, m0c, n0c);
        } else {
            cp.advance(w);
        }
    }
    cp_async_wait<0>();
    if (cl) cluster_sum_store<Cfg>(a, acc, smem, a_row0, b_col0, tid);
    // Lets a programmatic dependent launch (the stream-K reduction) get scheduled
    // now; it still waits for this whole grid to finish before reading results.
    asm volatile("griddepcontrol.launch_dependents;");
}

template <class Cfg>
constexpr KernelEntry make_entry(const char* name) {
    return KernelEntry{name,
                       reinterpret_cast<const void*>(&sgemm_ffma_kernel<Cfg>),
                       Cfg::BM, Cfg::BN, Cfg::BK, Cfg::WM, Cfg::WN, Cfg::TM, Cfg::TN,
                       Cfg::STAGES, Cfg::NT, Cfg::SMEM_BYTES, Cfg::VEC, Cfg::FMA2 ? 1 : 0, 0};
}

}  // namespace sgemm
