// Tile-table entries with 4-byte global loads: any pointer alignment and any
// leading dimension (e.g. odd lda / ldb).
#include "sgemm_ffma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB>
using W256V1 = FfmaCfg<128, 256, 32, 8, 16, 4, 4, 2, 3, 1, 4, true, 1>;
using Big16x8V1 = FfmaCfg<128, 128, 16, 16, 8, 4, 2, 2, 4, 1, 4, true, 2>;
using Small8x8V1 = FfmaCfg<64, 64, 16, 8, 8, 4, 2, 1, 3, 1, 4, true, 4>;

static const KernelEntry kEntries[] = {
    make_entry<W256V1>("128x256x32_t8x16_s3_f2_v1"),
    make_entry<Big16x8V1>("128x128x16_t16x8_s4_f2_v1"),
    make_entry<Small8x8V1>("64x64x16_t8x8_s3_f2_v1"),
};

const KernelEntry* ffma_entries_any(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
