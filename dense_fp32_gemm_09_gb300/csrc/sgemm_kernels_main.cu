// Tile-table entries with 16-byte global loads (rows 16-byte aligned): the
// large-tile FFMA2 kernels.
#include "sgemm_ffma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB, PIPE, KU,
//         SPREAD, SPREAD_FRAC>
// One 256-thread CTA per SM with 8 x 16 register tiles (up to 255 registers): the
// large-problem workhorses; BK = 64 halves the per-slice overhead when K is long.
// SPREAD issues the next slice's copies of an interior tile in that many parts at
// evenly spaced k-steps of the first 1 / SPREAD_FRAC of the current slice, instead
// of one burst before it (sgemm_ffma.cuh, compute_slice).  Same box, interleaved
// (TFLOP/s at 4096^3 / 8192^3 / 2048^3):
//   * 128 x 256 x 64, fragments double-buffered (A two k at a time): one burst
//     61.4 / 62.3 / 55.5; 4 parts over the whole slice 65.3 / 66.4 / 58.5; over
//     its first half 65.1 / 66.2; over its first quarter (every 4 k) 66.0 / 67.2 /
//     58.9; 8 parts over a quarter 64.9 / 66.1; 2 parts 63.8-64.3;
//   * 256 x 128 x 64, the eight 32 x 128 warp tiles stacked along M, slice loop
//     unrolled over half a slice: one burst 61.9 / 62.6 / 57.3; 8 parts over the
//     slice 64.0 / 64.8 / 59.4; 4 over its first half 64.5 / 65.2 / 59.5;
//   * 128 x 256 x 32 and 256 x 128 x 32, 4 stages, 8 parts over the slice: 1536^3
//     51.1 (256 x 128, one burst) -> 53.4 and 52.6; 1024^3 unchanged.
using W256K64 = FfmaCfg<128, 256, 64, 8, 16, 4, 4, 2, 2, 4, 2, true, 1, true, 0, 4, 4>;
using W256K32 = FfmaCfg<128, 256, 32, 8, 16, 4, 4, 2, 4, 4, 4, true, 1, false, 0, 8>;
using W256K16 = FfmaCfg<128, 256, 16, 8, 16, 4, 4, 2, 6, 4, 4, true, 1>;
using H256K64 = FfmaCfg<256, 128, 64, 8, 16, 4, 8, 1, 2, 4, 4, true, 1, false, 8, 4, 2>;
// The same tile with every refill in one burst: tiles that cross M or N refill in
// one bounds-checked burst either way, and with under 1.5 waves of tiles the CTAs
// holding them set the pace; there the all-burst twin measured faster (3008 x 2048
// x 2048: 57.7 against 56.4 TFLOP/s; 3004 x 2048 x 2000: 55.9 against 55.0), while
// at 1.8 waves and more the spread one leads (2900^3: 55.9 against 55.2).
using H256K64B = FfmaCfg<256, 128, 64, 8, 16, 4, 8, 1, 2, 4, 4, true, 1, false, 8>;
using H256K32 = FfmaCfg<256, 128, 32, 8, 16, 4, 8, 1, 4, 4, 4, true, 1, false, 0, 8>;
// Two CTAs per SM with 8 x 8 tiles (128 registers).
using S128K32 = FfmaCfg<128, 128, 32, 8, 8, 4, 4, 2, 3, 4, 4, true, 2>;
// Scalar-FFMA counterpart of the same tile, kept for comparison with fma.rn.f32x2.
using S128F1 = FfmaCfg<128, 128, 16, 8, 8, 4, 4, 2, 4, 4, 4, false, 2>;

static const KernelEntry kEntries[] = {
    make_entry<W256K64>("128x256x64_t8x16_s2_f2_v4"),
    make_entry<W256K32>("128x256x32_t8x16_s4_f2_v4"),
    make_entry<W256K16>("128x256x16_t8x16_s6_f2_v4"),
    make_entry<H256K64>("256x128x64_t8x16_s2_f2_v4"),
    make_entry<H256K64B>("256x128x64_t8x16_s2_f2_v4_burst"),
    make_entry<H256K32>("256x128x32_t8x16_s4_f2_v4"),
    make_entry<S128K32>("128x128x32_t8x8_s3_f2_v4"),
    make_entry<S128F1>("128x128x16_t8x8_s4_f1_v4"),
};

const KernelEntry* ffma_entries_main(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
