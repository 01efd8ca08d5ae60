// Tile-table entries with 16-byte global loads (rows 16-byte aligned): the
// large-tile FFMA2 kernels.
#include "sgemm_ffma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB, PIPE, KU,
//         SPREAD>
// One 256-thread CTA per SM with 8 x 16 register tiles (up to 255 registers): the
// large-problem workhorses; BK = 64 halves the per-slice overhead when K is long.
// SPREAD issues the next slice's copies of an interior tile in that many parts
// spaced over the current slice instead of one burst (sgemm_ffma.cuh,
// compute_slice); same box, interleaved, against one burst:
//   * 128 x 256 x 64, fragments double-buffered (A two k at a time), 4 parts:
//     4096^3 61.4 -> 65.4 TFLOP/s, 8192^3 62.3 -> 66.5;
//   * 256 x 128 x 64, the eight 32 x 128 warp tiles stacked along M, slice loop
//     unrolled over half a slice, 8 parts: 4096^3 61.9 -> 64.1, 2048^3 57.3 ->
//     59.4 (where the double-buffered entry reaches 58.5);
//   * 128 x 256 x 32 and 256 x 128 x 32, 4 stages, 8 parts: 1536^3 51.1 (256 x 128,
//     one burst) -> 53.4 and 52.6; 1024^3 unchanged.
using W256K64 = FfmaCfg<128, 256, 64, 8, 16, 4, 4, 2, 2, 4, 2, true, 1, true, 0, 4>;
using W256K32 = FfmaCfg<128, 256, 32, 8, 16, 4, 4, 2, 4, 4, 4, true, 1, false, 0, 8>;
using W256K16 = FfmaCfg<128, 256, 16, 8, 16, 4, 4, 2, 6, 4, 4, true, 1>;
using H256K64 = FfmaCfg<256, 128, 64, 8, 16, 4, 8, 1, 2, 4, 4, true, 1, false, 8, 8>;
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
    make_entry<H256K32>("256x128x32_t8x16_s4_f2_v4"),
    make_entry<S128K32>("128x128x32_t8x8_s3_f2_v4"),
    make_entry<S128F1>("128x128x16_t8x8_s4_f1_v4"),
};

const KernelEntry* ffma_entries_main(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
