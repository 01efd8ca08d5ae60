// Tile-table entries fed by TMA (16-byte-aligned operands, leading dimensions
// that are multiples of 4).
#include "sgemm_ffma_tma.cuh"

namespace sgemm {

// FfmaCfg<BM, BN, BK, TM, TN, LR, WARPS_M, WARPS_N, STAGES, VEC, AK, FMA2, MINB>
using Tma256K64 = FfmaCfg<128, 256, 64, 8, 16, 4, 4, 2, 2, 4, 2, true, 1>;
using Tma256K32 = FfmaCfg<128, 256, 32, 8, 16, 4, 4, 2, 4, 4, 2, true, 1>;
using TmaH256K32 = FfmaCfg<256, 128, 32, 8, 16, 4, 8, 1, 4, 4, 2, true, 1>;

static const KernelEntry kEntries[] = {
    make_tma_entry<Tma256K64>("128x256x64_t8x16_s2_f2_tma"),
    make_tma_entry<Tma256K32>("128x256x32_t8x16_s4_f2_tma"),
    make_tma_entry<TmaH256K32>("256x128x32_t8x16_s4_f2_tma"),
};

const KernelEntry* ffma_entries_tma(int* count) {
    *count = static_cast<int>(sizeof(kEntries) / sizeof(kEntries[0]));
    return kEntries;
}

}  // namespace sgemm
