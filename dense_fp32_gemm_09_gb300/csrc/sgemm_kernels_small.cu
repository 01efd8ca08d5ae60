// Tile-table entries with 16-byte global loads for small or narrow problems.
#include "sgemm_ffma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB, PIPE, KU,
//         SPREAD>
using Tall16x8 = FfmaCfg<128, 64, 16, 16, 8, 4, 2, 1, 4, 4, 4, true, 4>;
// One 256-thread CTA per SM for narrow C (N <= 64): eight 64 x 64 warp tiles
// stacked along M, 8 x 16 register tiles with 8 lane-rows.  With four 64-thread
// CTAs per SM instead, the warp scheduler lets some CTAs run ahead and the SM
// spends the last third of a 16384 x 64 x 4096 product short of warps.
// Its next slice's copies go out in 4 parts over the first half of the current one
// (sgemm_ffma.cuh, compute_slice), and its fragments are double-buffered (A two k at
// a time).  Same box, TFLOP/s at 16384 x 64 x 4096 / 8192 x 64 x 8192 / 4096 x 64 x
// 4096: one burst 50.3 / - / -; 4 parts, single-buffered 52.4 / 52.9 / 39.8; 4 parts
// over the first half, double-buffered 53.6 / 53.8 / 41.4 (2 or 8 parts, or the first
// quarter, slower).
using Tall512K32 = FfmaCfg<512, 64, 32, 8, 16, 8, 8, 1, 2, 4, 2, true, 1, true, 0, 4, 2>;
// The next slice's copies in 4 parts over the current one: 768^3 25.5 -> 27.1
// TFLOP/s, 2048 x 64 x 4096 28.6 -> 30.3, 512^3 unchanged (same box).
using Small8x8 = FfmaCfg<64, 64, 16, 8, 8, 4, 2, 1, 3, 4, 4, true, 4, false, 0, 4>;
using Small4x4 = FfmaCfg<64, 64, 16, 4, 4, 4, 4, 2, 3, 4, 4, false, 3>;
using Small8x4 = FfmaCfg<64, 64, 16, 8, 4, 4, 2, 2, 3, 4, 4, true, 4>;
using Tiny4x4 = FfmaCfg<32, 32, 16, 4, 4, 4, 2, 1, 3, 4, 4, true, 8>;

static const KernelEntry kEntries[] = {
    make_entry<Tall16x8>("128x64x16_t16x8_s4_f2_v4"),
    make_entry<Tall512K32>("512x64x32_t8x16_s2_f2_v4"),
    make_entry<Small8x8>("64x64x16_t8x8_s3_f2_v4"),
    make_entry<Small4x4>("64x64x16_t4x4_s3_f1_v4"),
    make_entry<Small8x4>("64x64x16_t8x4_s3_f2_v4"),
    make_entry<Tiny4x4>("32x32x16_t4x4_s3_f2_v4"),
};

const KernelEntry* ffma_entries_small(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
