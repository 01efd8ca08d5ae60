"""The per-shape tile table as host logic (no GPU).

sgemm_choose_check runs the same rules sgemm_run applies before any launch, for a
given SM count and operand alignment.  Each case below sits on one rule, and the
neighbouring cases sit just across its boundary, so a changed threshold or a
reordered rule fails here rather than only as a slower run."""
import ctypes

import pytest

GB300_SMS = 152


def _choose(lib, M, N, K, lda=None, ldb=None, a_off=0, b_off=0, sms=GB300_SMS):
    kid, packed = ctypes.c_int(-7), ctypes.c_int(-7)
    rc = lib.sgemm_choose_check(M, N, K, K if lda is None else lda, N if ldb is None else ldb,
                                a_off, b_off, sms, ctypes.byref(kid), ctypes.byref(packed))
    assert rc == 0, (M, N, K, lib.sgemm_last_error())
    return lib.sgemm_kernel_name(kid.value).decode(), packed.value


@pytest.mark.parametrize("shape,expected", [
    # 64-deep slices on 128 x 256 tiles with double-buffered fragments once every
    # CTA gets at least 44 of them (tiles of 128 x 256 times 64-deep slices a tile,
    # over 152 SMs) ...
    ((4096, 4096, 4096), "128x256x64_t8x16_s2_f2_v4"),
    ((8192, 8192, 8192), "128x256x64_t8x16_s2_f2_v4"),
    ((4864, 4864, 2048), "128x256x64_t8x16_s2_f2_v4"),  # 722 tiles * 32 / 152 = 152
    ((1920, 4864, 2048), "128x256x64_t8x16_s2_f2_v4"),  # 285 * 32 / 152 = 60
    ((4096, 4096, 2044), "128x256x64_t8x16_s2_f2_v4"),  # 512 * 32 / 152 = 107
    ((4096, 4096, 1536), "128x256x64_t8x16_s2_f2_v4"),  # 512 * 24 / 152 = 80
    ((8192, 8192, 512), "128x256x64_t8x16_s2_f2_v4"),   # 2048 * 8 / 152 = 107
    ((3072, 3072, 1536), "128x256x64_t8x16_s2_f2_v4"),  # 288 * 24 / 152 = 45
    # ... else 64-deep slices on 256 x 128 tiles once every CTA gets about 16 of
    # them (tiles of 256 x 128 times 64-deep slices a tile, over 152 SMs) ...
    ((2048, 2048, 2048), "256x128x64_t8x16_s2_f2_v4"),  # 128 * 32 / 152 = 26
    ((2560, 2560, 1280), "256x128x64_t8x16_s2_f2_v4"),  # 200 * 20 / 152 = 26
    ((4096, 4096, 768), "256x128x64_t8x16_s2_f2_v4"),   # 512 * 12 / 152 = 40
    # ... else 32-deep slices on 128 x 256 tiles (1024^3: 4*8*16 = 512 64-deep
    # slices; 1536^3: 1728).
    ((1024, 1024, 1024), "128x256x32_t8x16_s4_f2_v4"),
    ((1536, 1536, 1536), "128x256x32_t8x16_s4_f2_v4"),
    ((1024, 2048, 2044), "128x256x32_t8x16_s4_f2_v4"),  # 4*16*32 = 2048 < 16*152
    ((1536, 2048, 2044), "256x128x64_t8x16_s2_f2_v4"),  # 6*16*32 = 3072 >= 16*152
    ((896, 768, 2048), "128x256x32_t8x16_s4_f2_v4"),    # K = 2048 but 4*6*32 = 768
    ((768, 1024, 2048), "128x256x32_t8x16_s4_f2_v4"),   # 3*8*32 = 768
    # Tiles crossing M or N with under 1.5 waves of 256 x 128 tiles: the all-burst twin.
    ((3008, 2048, 2048), "256x128x64_t8x16_s2_f2_v4_burst"),  # 12*16 = 192 < 228
    ((3500, 2048, 2048), "256x128x64_t8x16_s2_f2_v4_burst"),  # 14*16 = 224
    ((3584, 2048, 2048), "128x256x64_t8x16_s2_f2_v4"),        # no tile crosses: 47 a CTA
    ((3600, 2048, 2048), "128x256x64_t8x16_s2_f2_v4"),        # 15*16 = 240 tiles: 48 a CTA
    ((2816, 2048, 2048), "256x128x64_t8x16_s2_f2_v4"),        # 11*16 tiles, 41 a CTA
    ((2048, 2000, 2048), "256x128x64_t8x16_s2_f2_v4_burst"),  # N edge, 8*16 tiles
    # The smallest problems: at most SMs/4 tiles of 64 x 64 and K <= 1024.
    ((256, 256, 256), "32x32x16_t4x4_s3_f2_v4"),
    ((384, 384, 384), "32x32x16_t4x4_s3_f2_v4"),
    ((384, 384, 1024), "32x32x16_t4x4_s3_f2_v4"),
    ((384, 384, 1028), "64x64x16_t8x8_s3_f2_v4"),    # K too deep: few 128 tiles -> 64 x 64
    ((448, 384, 384), "64x64x16_t8x8_s3_f2_v4"),     # 42 tiles of 64^2: 168 > 152
    ((256, 256, 2048), "64x64x16_t8x8_s3_f2_v4"),    # 4 tiles of 128^2: 64 x 64 stays
    # Small C (fewer than SMs/4 tiles of 128^2) with K >= 2048: 128 x 256 tiles from 8
    # of them with at most a quarter to spare or from 4 with at most a tenth, else
    # 128 x 128 from 9 with at most a fifth.
    ((384, 384, 2048), "128x128x32_t8x8_s3_f2_v4"),   # 6 wide tiles, 25 % spare: 128^2
    ((448, 448, 4096), "128x256x32_t8x16_s4_f2_v4"),  # 8 wide tiles, 23 % spare
    ((512, 512, 2048), "128x256x32_t8x16_s4_f2_v4"),  # 8 wide tiles, none spare
    ((256, 512, 8192), "128x256x32_t8x16_s4_f2_v4"),  # 4 wide tiles
    ((640, 640, 4096), "128x256x32_t8x16_s4_f2_v4"),  # 15 wide tiles, 17 % spare
    ((768, 768, 8192), "128x256x32_t8x16_s4_f2_v4"),
    ((320, 320, 4096), "64x64x16_t8x8_s3_f2_v4"),     # both larger tiles a third empty
    ((768, 768, 2044), "64x64x16_t8x8_s3_f2_v4"),     # K below 2048
    # Narrow C (N <= 64): 512-row tiles once M >= 2560, else 64 x 64.
    ((16384, 64, 4096), "512x64x32_t8x16_s2_f2_v4"),
    ((4096, 36, 100), "512x64x32_t8x16_s2_f2_v4"),
    ((3000, 64, 3000), "512x64x32_t8x16_s2_f2_v4"),
    ((2560, 64, 4096), "512x64x32_t8x16_s2_f2_v4"),
    ((2559, 64, 4096), "64x64x16_t8x8_s3_f2_v4"),
    ((2000, 64, 2048), "64x64x16_t8x8_s3_f2_v4"),
    # 64 < N <= 128 with M >= 4096: the 128-wide tile, 64-deep from 4 of its 64-deep
    # slices a CTA, 32-deep from 1.25, else 128 x 128 tiles.
    ((8192, 128, 4096), "256x128x64_t8x16_s2_f2_v4"),   # 32 * 64 = 2048 slices
    ((4096, 96, 2432), "256x128x64_t8x16_s2_f2_v4"),    # 16 * 38 = 608 = 4 * 152
    ((4096, 96, 2368), "256x128x32_t8x16_s4_f2_v4"),    # 16 * 37 = 592
    ((8192, 128, 1024), "256x128x32_t8x16_s4_f2_v4"),   # 32 * 16 = 512
    ((4096, 128, 768), "256x128x32_t8x16_s4_f2_v4"),    # 16 * 12 = 192 >= 190
    ((4096, 128, 704), "128x128x32_t8x8_s3_f2_v4"),     # 16 * 11 = 176
    ((4096, 128, 512), "128x128x32_t8x8_s3_f2_v4"),
    ((8192, 96, 64), "128x128x32_t8x8_s3_f2_v4"),
    # N <= 256 that 64-wide tiles fit more closely than 128-wide ones, M >= 4096.
    ((8192, 192, 4096), "512x64x32_t8x16_s2_f2_v4"),
    ((8192, 160, 1024), "512x64x32_t8x16_s2_f2_v4"),
    ((8192, 256, 4096), "256x128x64_t8x16_s2_f2_v4"),   # both fit: 2 x 128
    ((4000, 192, 4096), "128x256x32_t8x16_s4_f2_v4"),   # M below 4096: general rules
    # Short, wide C (M <= 64): tiles no taller than C.
    ((64, 8192, 4096), "64x64x16_t8x8_s3_f2_v4"),
    ((48, 4096, 1024), "64x64x16_t8x8_s3_f2_v4"),
    ((32, 16384, 4096), "32x32x16_t4x4_s3_f2_v4"),
    ((96, 4096, 4096), "128x256x32_t8x16_s4_f2_v4"),    # M above 64: small-C rules
    # Small C with N <= 128: the 256 x 128 orientation.
    ((2048, 128, 2048), "256x128x32_t8x16_s4_f2_v4"),
    # Below M = 4096 that rule yields: 32 tiles of 128^2 are fewer than SMs/4.
    ((4095, 128, 1024), "64x64x16_t8x8_s3_f2_v4"),
    ((2048, 256, 1024), "64x64x16_t8x8_s3_f2_v4"),     # 32 tiles of 128^2
    ((4096, 256, 1024), "128x256x32_t8x16_s4_f2_v4"),  # 64 tiles of 128^2: 256 > 152
])
def test_rules_for_aligned_operands(lib, shape, expected):
    assert _choose(lib, *shape) == (expected, 0)


def test_sm_count_moves_the_thresholds(lib):
    # 13 SMs: 1024^3 has 512 >= 20*13 deep slices; 256^3 is no longer "few tiles".
    assert _choose(lib, 1024, 1024, 1024, sms=13)[0] == "256x128x64_t8x16_s2_f2_v4"
    assert _choose(lib, 256, 256, 256, sms=13)[0] == "128x256x32_t8x16_s4_f2_v4"
    # 13 SMs: 2048^3 has 128 tiles of 128 x 256, more than two waves of 13.
    assert _choose(lib, 2048, 2048, 2048, sms=13)[0] == "128x256x64_t8x16_s2_f2_v4"
    # Many SMs: 1024^3 has 256 tiles of 64^2, within SMs/4 at 1024 SMs.
    assert _choose(lib, 1024, 1024, 1024, sms=1024)[0] == "32x32x16_t4x4_s3_f2_v4"
    assert _choose(lib, 1024, 1024, 1024, sms=1023)[0] == "64x64x16_t8x8_s3_f2_v4"


def test_misaligned_operands_small_products_take_scalar_loads(lib):
    # Below 5e8 multiply-adds, or with K < 768, nothing is packed: 4-byte loads.
    assert _choose(lib, 700, 700, 1000, lda=1001) == ("128x128x16_t16x8_s4_f2_v1", 0)  # 4.9e8
    assert _choose(lib, 1000, 1000, 300, lda=301) == ("128x128x16_t16x8_s4_f2_v1", 0)  # 64 tiles
    assert _choose(lib, 1500, 1500, 700, lda=701) == ("128x256x32_t8x16_s3_f2_v1", 0)  # 144 tiles
    assert _choose(lib, 512, 512, 512, lda=513) == ("64x64x16_t8x8_s3_f2_v1", 0)       # 16 tiles
    assert _choose(lib, 4096, 64, 300, lda=301) == ("64x64x16_t8x8_s3_f2_v1", 0)      # N = 64
    assert _choose(lib, 800, 800, 780, lda=781) == ("128x128x16_t16x8_s4_f2_v1", 0)  # 4.99e8
    assert _choose(lib, 300, 300, 300, ldb=301) == ("64x64x16_t8x8_s3_f2_v1", 0)
    assert _choose(lib, 4096, 4096, 767, lda=769)[1] == 0     # K just short of 768
    assert _choose(lib, 2048, 2048, 511, b_off=2)[1] == 0
    # The 16-byte-load-only rules do not apply without aligned operands.
    assert _choose(lib, 16384, 64, 100, lda=101) == ("128x256x32_t8x16_s3_f2_v1", 0)


def test_misaligned_operands_large_products_are_packed(lib):
    # K >= 768 and M*N*K >= 5e8: the misaligned operand alone is packed, then the
    # aligned rules apply.
    assert _choose(lib, 1000, 1000, 1000, lda=1001) == ("128x256x32_t8x16_s4_f2_v4", 1)
    assert _choose(lib, 1000, 1000, 1000, b_off=2) == ("128x256x32_t8x16_s4_f2_v4", 2)
    assert _choose(lib, 800, 800, 782, lda=783)[1] == 1     # 5.0e8
    assert _choose(lib, 4096, 4096, 768, lda=769)[1] == 1
    assert _choose(lib, 1291, 1292, 1292, lda=1293) == ("128x256x32_t8x16_s4_f2_v4", 1)
    assert _choose(lib, 1292, 1292, 1292, b_off=1) == ("128x256x32_t8x16_s4_f2_v4", 2)
    # The ragged workload: odd leading dimensions everywhere, both packed.
    assert _choose(lib, 3001, 2047, 1999, lda=2001, ldb=2049) == ("256x128x64_t8x16_s2_f2_v4_burst",
                                                                 3)
    assert _choose(lib, 4096, 4096, 4096, a_off=3, b_off=1) == ("128x256x64_t8x16_s2_f2_v4", 3)


def test_chosen_entry_matches_operand_alignment(lib):
    # Whatever the shape, a 16-byte-load entry is chosen only for aligned (or packed) operands.
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    names = {lib.sgemm_kernel_name(i).decode(): i for i in range(lib.sgemm_num_kernels())}
    for M, N, K in [(1, 1, 1), (7, 9, 13), (64, 64, 16), (500, 70, 3000), (4096, 200, 64),
                    (1300, 1300, 1300), (33, 4096, 4096), (5000, 300, 33)]:
        for lda_pad, b_off in [(0, 0), (1, 0), (0, 3)]:
            name, packed = _choose(lib, M, N, K, lda=K + lda_pad, b_off=b_off)
            cfg = SgemmConfig()
            assert lib.sgemm_kernel_info(names[name], ctypes.byref(cfg)) == 0
            a_ok = lda_pad == 0 and K % 4 == 0 or packed & 1
            b_ok = b_off == 0 and N % 4 == 0 or packed & 2
            assert (cfg.vec == 4) == bool(a_ok and b_ok), (M, N, K, lda_pad, b_off, name)


def test_forced_kernel_variable_is_not_consulted(lib, monkeypatch):
    monkeypatch.setenv("SGEMM_FORCE_KERNEL", "64x64x16_t4x4_s3_f1_v4")
    assert _choose(lib, 4096, 4096, 4096)[0] == "128x256x64_t8x16_s2_f2_v4"


def test_invalid_arguments(lib):
    kid = ctypes.c_int()
    bad = [(0, 4, 4, 4, 4, 0, 0, 152), (4, 4, 4, 3, 4, 0, 0, 152), (4, 4, 4, 4, 3, 0, 0, 152),
           (4, 4, 4, 4, 4, 4, 0, 152), (4, 4, 4, 4, 4, 0, -1, 152), (4, 4, 4, 4, 4, 0, 0, 0)]
    for args in bad:
        assert lib.sgemm_choose_check(*args, ctypes.byref(kid), None) == -1, args
    assert lib.sgemm_choose_check(4, 4, 4, 4, 4, 0, 0, 152, None, None) == -1
    assert lib.sgemm_choose_check(4, 4, 4, 4, 4, 0, 0, 152, ctypes.byref(kid), None) == 0
