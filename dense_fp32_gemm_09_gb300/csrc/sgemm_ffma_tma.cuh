// TMA-fed variant of the FFMA kernel (16-byte-aligned operands).
//
// Same hierarchy, register micro-kernel, persistent schedule and epilogue as
// sgemm_ffma.cuh; what changes is how the BK-deep slices reach shared memory
// ("Register/Shared Memory Tiling", 공유 메모리 타일 로딩 and 더블 버퍼링: the
// cooperative tile load and the buffer swap):
//   * one thread issues the whole slice as TMA tensor copies: A as BK/32 boxes
//     of 32 (k) x BM rows with the 128-byte swizzle, B as one box of BN x BK
//     without swizzle; zero fill outside the matrices comes from TMA;
//   * each ring slot has a `full` mbarrier (TMA transaction bytes) and an
//     `empty` mbarrier (one arrival per warp after it has read the slot), so
//     warps are never held at a CTA-wide barrier between slices and no thread
//     spends issue slots on copy addresses.
// A fragments are read as float4 of 4 consecutive k from one row.  With the
// swizzle, the 16-byte chunk c of row r sits at chunk c ^ (r & 7); a thread's
// rows are a_row0 + 4 i, so r & 7 is lr for even i and lr ^ 4 for odd i, and the
// XOR reduces to one offset per 4-k step (oe) and oe ^ 16 floats.
#pragma once

#include "sgemm_async.cuh"
#include "sgemm_ffma.cuh"

namespace sgemm {

struct FfmaTmaParams {
    CUtensorMap ta;   // A: boxes of 32 (k) x BM rows, 128-byte swizzle
    CUtensorMap tb;   // B: boxes of BN (n) x BK rows, no swizzle
    GemmArgs g;
};

template <class Cfg>
struct TmaLayout {
    static constexpr int KH = Cfg::BK / 32;           // 32-wide k blocks of the A slice
    static constexpr int A_BLOCK = Cfg::BM * 32;      // floats of one A block
    static constexpr int A_STAGE = KH * A_BLOCK;
    static constexpr int B_STAGE = Cfg::BK * Cfg::BN;
    static constexpr int STAGE = A_STAGE + B_STAGE;   // floats per ring slot
    static constexpr uint32_t STAGE_BYTES = STAGE * 4;
    static constexpr int SMEM_BYTES = Cfg::STAGES * STAGE * 4 + 1024;  // + alignment slack
    static constexpr int NWARPS = Cfg::NT / 32;
    static_assert(Cfg::BK % 32 == 0, "BK must be a multiple of 32");
    static_assert(Cfg::LR == 4 && (Cfg::AK == 4 || Cfg::AK == 2) && Cfg::VEC == 4,
                  "layout assumptions");
    static_assert(Cfg::WM % 8 == 0, "warp rows must start on a swizzle period");
    static_assert((A_STAGE * 4) % 1024 == 0 && (STAGE * 4) % 1024 == 0, "1024-byte slots");
    static_assert(Cfg::BN <= 256 && Cfg::BK <= 256 && Cfg::BM <= 256, "TMA box limits");
};

// A fragments of AK consecutive k (one 16- or 8-byte load per row) from the
// swizzled A slice; B values of one k.
template <class Cfg>
__device__ __forceinline__ void load_a_frag_tma(const float* sA, int a_row0, int lr4, int kq,
                                                float (&av)[Cfg::TM][Cfg::AK]) {
    constexpr int BM = Cfg::BM, TM = Cfg::TM, LR = Cfg::LR, AK = Cfg::AK;
    const int h = kq / 32, c = (kq % 32) / 4, sub = kq % 4;
    const int oe = ((c * 4) ^ lr4) + sub;   // rows with r & 7 == lr
    const int oo = oe ^ 16;                 // rows with r & 7 == lr + 4
    const float* ah = sA + a_row0 * 32 + h * BM * 32;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const float* pa = ah + i * LR * 32 + ((i & 1) ? oo : oe);
        if constexpr (AK == 4) {
            const float4 t = *reinterpret_cast<const float4*>(pa);
            av[i][0] = t.x; av[i][1] = t.y; av[i][2] = t.z; av[i][3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2*>(pa);
            av[i][0] = t.x; av[i][1] = t.y;
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void load_b_frag_tma(const float* sB, int b_col0, int k,
                                                float4 (&b)[Cfg::TN / 4]) {
#pragma unroll
    for (int j4 = 0; j4 < Cfg::TN / 4; ++j4)
        b[j4] = *reinterpret_cast<const float4*>(sB + k * Cfg::BN + b_col0 + j4 * Cfg::LC * 4);
}

template <class Cfg, class AccT>
__device__ __forceinline__ void compute_slice_tma(const float* sA, const float* sB, int a_row0,
                                                  int lr4, int b_col0, AccT& acc) {
    constexpr int BK = Cfg::BK, TM = Cfg::TM, TN = Cfg::TN, AK = Cfg::AK;
#pragma unroll
    for (int kq = 0; kq < BK; kq += AK) {
        float av[TM][AK];
        load_a_frag_tma<Cfg>(sA, a_row0, lr4, kq, av);
#pragma unroll
        for (int kk = 0; kk < AK; ++kk) {
            float4 b[TN / 4];
            load_b_frag_tma<Cfg>(sB, b_col0, kq + kk, b);
            float ak[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i) ak[i] = av[i][kk];
            acc.rank1(ak, b);
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void tma_issue_slice(const FfmaTmaParams& P, uint32_t slot_addr,
                                                uint32_t full_bar, int m0, int n0, int k0) {
    using L = TmaLayout<Cfg>;
    async::mbar_expect_tx(full_bar, L::STAGE_BYTES);
#pragma unroll
    for (int h = 0; h < L::KH; ++h)
        async::tma_load_2d(slot_addr + h * L::A_BLOCK * 4, &P.ta, k0 + 32 * h, m0, full_bar);
    async::tma_load_2d(slot_addr + L::A_STAGE * 4, &P.tb, n0, k0, full_bar);
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MINB)
    sgemm_ffma_tma_kernel(const __grid_constant__ FfmaTmaParams P) {
    using L = TmaLayout<Cfg>;
    using AccT = Acc<Cfg::TM, Cfg::TN, Cfg::FMA2, false>;
    constexpr int STAGES = Cfg::STAGES, BK = Cfg::BK;
    const GemmArgs& a = P.g;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ int abort_s;
    float* const smem = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem0 = async::su32(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int warp_m = warp / Cfg::WARPS_N, warp_n = warp % Cfg::WARPS_N;
    constexpr int LRQ = Cfg::LR < 8 ? Cfg::LR : 8;
    constexpr int LCQ = 8 / LRQ;
    const int q = lane >> 3, li = lane & 7;
    const int lr = (q % (Cfg::LR / LRQ)) * LRQ + li % LRQ;
    const int lc = (q / (Cfg::LR / LRQ)) * LCQ + li / LRQ;
    const int a_row0 = warp_m * Cfg::WM + lr;
    const int b_col0 = warp_n * Cfg::WN + lc * 4;

    // The CTA's work description and the loader cursor (thread 0 only) live in
    // shared memory: every register goes to the accumulators and fragments.
    __shared__ CtaWork s_w;
    __shared__ Cursor s_ld;
    if (tid == 0) {
        s_w = make_work(a, blockIdx.x);
        for (int s = 0; s < STAGES; ++s) {
            async::mbar_init(async::su32(&full_bar[s]), 1);
            async::mbar_init(async::su32(&empty_bar[s]), L::NWARPS);
        }
        abort_s = 0;
        async::mbar_fence_init();
        // Programmatic dependent launch: the first global read waits for the
        // stream's previous kernel to complete.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        Cursor ld;   // next slice to load; ld.c = slices issued so far
        ld.seek(s_w, 0);
        for (int s = 0; s < STAGES && ld.c < s_w.total; ++s) {
            int m0, n0;
            tile_origin(a, ld.tile, Cfg::BM, Cfg::BN, m0, n0);
            tma_issue_slice<Cfg>(P, smem0 + s * L::STAGE_BYTES, async::su32(&full_bar[s]), m0, n0,
                                 ld.kt * BK);
            ld.advance(s_w);
        }
        s_ld = ld;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");   // (returns at once by now)
    const CtaWork& w = s_w;
    if (w.total <= 0) return;
    volatile int* abort_flag = &abort_s;
    Cursor cp;
    cp.seek(w, 0);

    AccT acc;
    acc.zero();
    int m0c, n0c;
    tile_origin(a, cp.tile, Cfg::BM, Cfg::BN, m0c, n0c);
    int s = 0;          // ring slot of slice cp.c
    uint32_t par = 0;   // phase parity of that slot's barriers
    bool ok = true;
    while (cp.c < w.total) {
        if (!async::mbar_wait(async::su32(&full_bar[s]), par, abort_flag, a.status)) {
            ok = false;
            break;
        }
        compute_slice_tma<Cfg>(smem + s * L::STAGE, smem + s * L::STAGE + L::A_STAGE, a_row0,
                               lr * 4, b_col0, acc);
        __syncwarp();
        if (lane == 0) async::mbar_arrive(async::su32(&empty_bar[s]));
        // Refill this slot once every warp has read it.
        if (tid == 0 && s_ld.c < w.total) {
            if (!async::mbar_wait(async::su32(&empty_bar[s]), par, abort_flag, a.status)) {
                ok = false;
                break;
            }
            Cursor ld = s_ld;
            int m0, n0;
            tile_origin(a, ld.tile, Cfg::BM, Cfg::BN, m0, n0);
            tma_issue_slice<Cfg>(P, smem0 + s * L::STAGE_BYTES, async::su32(&full_bar[s]), m0,
                                 n0, ld.kt * BK);
            ld.advance(w);
            s_ld = ld;
        }
        if (cp.kt + 1 == cp.kt_end) {
            if (cp.kt_begin == 0 && cp.kt_end == w.KT)
                store_tile<Cfg>(a, acc, m0c, n0c, a_row0, b_col0);
            else
                store_partial<Cfg>(a, w, cp, acc, a_row0, b_col0);
            acc.zero();
            cp.advance(w);
            if (cp.c < w.total) tile_origin(a, cp.tile, Cfg::BM, Cfg::BN, m0c, n0c);
        } else {
            cp.advance(w);
        }
        if (++s == STAGES) {
            s = 0;
            par ^= 1u;
        }
    }
    if (!ok && tid == 0) {
        // Gave up: let the copies still in flight land before the CTA exits.
        volatile int no_abort = 0;
        for (long long j = cp.c; j < s_ld.c; ++j)
            async::mbar_wait(async::su32(&full_bar[j % STAGES]),
                             static_cast<uint32_t>((j / STAGES) & 1), &no_abort, nullptr);
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

template <class Cfg>
constexpr KernelEntry make_tma_entry(const char* name) {
    return KernelEntry{name,
                       reinterpret_cast<const void*>(&sgemm_ffma_tma_kernel<Cfg>),
                       Cfg::BM, Cfg::BN, Cfg::BK, Cfg::WM, Cfg::WN, Cfg::TM, Cfg::TN,
                       Cfg::STAGES, Cfg::NT, TmaLayout<Cfg>::SMEM_BYTES, Cfg::VEC,
                       Cfg::FMA2 ? 1 : 0, 1};
}

}  // namespace sgemm
