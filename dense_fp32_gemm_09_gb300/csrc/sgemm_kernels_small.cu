// Tile-table entries with 16-byte global loads for small or narrow problems.
#include "sgemm_ffma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB>
using Tall16x8 = FfmaCfg<128, 64, 16, 16, 8, 4, 2, 1, 4, 4, 4, true, 4>;
using Small8x8 = FfmaCfg<64, 64, 16, 8, 8, 4, 2, 1, 3, 4, 4, true, 4>;
using Small4x4 = FfmaCfg<64, 64, 16, 4, 4, 4, 4, 2, 3, 4, 4, false, 3>;
using Small8x4 = FfmaCfg<64, 64, 16, 8, 4, 4, 2, 2, 3, 4, 4, true, 4>;

static const KernelEntry kEntries[] = {
    make_entry<Tall16x8>("128x64x16_t16x8_s4_f2_v4"),
    make_entry<Small8x8>("64x64x16_t8x8_s3_f2_v4"),
    make_entry<Small4x4>("64x64x16_t4x4_s3_f1_v4"),
    make_entry<Small8x4>("64x64x16_t8x4_s3_f2_v4"),
};

const KernelEntry* ffma_entries_small(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
