"""Host-side checks of the persistent / stream-K schedule (no GPU).

sgemm_schedule_check plans a problem for a given SM count and residency and
walks every CTA's k-slice list with the same code the kernel runs."""
import ctypes
import itertools

import pytest

SHAPES = [(1, 1, 1), (3, 5, 7), (64, 64, 16), (65, 63, 17), (129, 127, 300), (256, 256, 256),
          (1, 1, 100000), (64, 64, 300000), (300, 1, 65536),
          (1024, 1024, 1024), (3001, 2047, 1999), (4096, 4096, 4096), (16384, 64, 4096),
          (8192, 8192, 8192), (5000, 300, 33), (128, 128, 100000)]
MACHINES = [(152, 1), (152, 2), (152, 3), (148, 2), (7, 1), (1, 1), (13, 4)]


def _cfg():
    from dense_fp32_gemm_09_gb300._abi import SgemmConfig
    return SgemmConfig()


@pytest.mark.parametrize("schedule", [0, 1, 2])
def test_schedule_covers_each_slice_once(lib, schedule):
    n = lib.sgemm_num_kernels()
    for kid, (M, N, K), (sms, occ) in itertools.product(range(n), SHAPES, MACHINES):
        cfg = _cfg()
        rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, schedule, ctypes.byref(cfg))
        assert rc == 0, (kid, M, N, K, sms, occ, schedule, lib.sgemm_last_error())
        assert cfg.grid <= sms * occ
        assert cfg.tiles == -(-M // cfg.bm) * -(-N // cfg.bn)
        if schedule == 1:
            assert cfg.sk_tiles == 0 and cfg.split_k == 1
        if cfg.sk_tiles > 0 and cfg.cluster == 0:
            # Stream-K shares its split tiles among more CTAs than there are such
            # tiles, so the reduction launch always has partial tiles to sum.
            assert cfg.sk_tiles < cfg.grid and cfg.split_k >= 2, (kid, M, N, K, sms, occ)


def test_stream_k_balances_a_partial_last_wave(lib):
    # 4096^3 with 128x256 tiles: 512 tiles on 152 resident CTAs -> 3 full waves
    # plus 56 tiles shared out by k-slices.
    table = [lib.sgemm_kernel_name(i).decode() for i in range(lib.sgemm_num_kernels())]
    kid = table.index("128x256x64_t8x16_s2_f2_v4")
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 4096, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (512, 152, 512 - 3 * 152)
    assert cfg.split_k >= 2
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 4096, kid, 152, 1, 1, ctypes.byref(cfg)) == 0
    assert cfg.sk_tiles == 0 and cfg.grid == 152


def test_partial_last_wave_goes_to_stream_k_when_that_shortens_it(lib):
    """Past whole waves, the leftover tiles are shared by k-slices when every CTA gets
    one and the shared tail, plus about two slices of stores and reduction, is
    shorter than another wave of whole tiles."""
    kid = _kid(lib, "128x256x64_t8x16_s2_f2_v4")
    # 4096 x 4096 x 512: 512 tiles = 3 waves + 56 tiles of 8 slices; 448 slices give
    # every CTA 3, and 3 + 2 < 8.
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 512, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (512, 152, 56) and cfg.split_k >= 2
    # 4 slices a tile: 224 slices give 2 a CTA, and 2 + 2 is not shorter than 4.
    cfg = _cfg()
    assert lib.sgemm_schedule_check(4096, 4096, 256, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (512, 152, 0)
    # 153 tiles of 64 slices: the one leftover tile has fewer slices than CTAs.
    cfg = _cfg()
    assert lib.sgemm_schedule_check(9 * 128, 17 * 256, 4096, kid, 152, 1, 0,
                                    ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (153, 152, 0)
    # 155 tiles of 64 slices: 192 leftover slices, 2 a CTA: shared.
    cfg = _cfg()
    assert lib.sgemm_schedule_check(5 * 128, 31 * 256, 4096, kid, 152, 1, 0,
                                    ctypes.byref(cfg)) == 0
    assert (cfg.tiles, cfg.grid, cfg.sk_tiles) == (155, 152, 3)


def test_small_problem_splits_k(lib, monkeypatch):
    monkeypatch.setenv("SGEMM_CLUSTER", "0")   # the stream-K form of the split
    table = [lib.sgemm_kernel_name(i).decode() for i in range(lib.sgemm_num_kernels())]
    kid = table.index("128x256x32_t8x16_s4_f2_v4")
    cfg = _cfg()
    assert lib.sgemm_schedule_check(1024, 1024, 1024, kid, 152, 1, 0, ctypes.byref(cfg)) == 0
    assert cfg.tiles == 32 and cfg.sk_tiles == 32 and cfg.grid == 152


def test_rejects_bad_arguments(lib):
    assert lib.sgemm_schedule_check(0, 4, 4, 0, 152, 2, 0, None) == -1
    assert lib.sgemm_schedule_check(4, 4, 4, 0, 0, 2, 0, None) == -1
    assert lib.sgemm_schedule_check(4, 4, 4, 999, 152, 2, 0, None) == -1


@pytest.mark.parametrize("M,N,K", [(67000, 64, 32768), (50000, 45000, 8)])
def test_schedule_of_operands_past_2_31_elements(lib, M, N, K):
    """The shapes of the GPU tests whose A or C hold more than 2**31 elements."""
    for kid in range(lib.sgemm_num_kernels()):
        for sms, occ in [(152, 1), (152, 4)]:
            cfg = _cfg()
            rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, 0, ctypes.byref(cfg))
            assert rc == 0, (kid, sms, occ, lib.sgemm_last_error())


# --------------------------------------------------------------------------
# stream-K gap: split tiles separated by virtual slices that stand for the
# cost of one more partial-tile store
# --------------------------------------------------------------------------


def _kid(lib, name):
    return [lib.sgemm_kernel_name(i).decode()
            for i in range(lib.sgemm_num_kernels())].index(name)


@pytest.mark.parametrize("gap", [1, 2, 3])
@pytest.mark.parametrize("schedule", [0, 2])
def test_forced_gap_covers_each_slice_once(lib, monkeypatch, gap, schedule):
    monkeypatch.setenv("SGEMM_SK_GAP", str(gap))
    n = lib.sgemm_num_kernels()
    used = 0
    for kid, (M, N, K), (sms, occ) in itertools.product(range(n), SHAPES, MACHINES):
        cfg = _cfg()
        rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, schedule, ctypes.byref(cfg))
        assert rc == 0, (kid, M, N, K, sms, occ, gap, lib.sgemm_last_error())
        assert cfg.sk_gap in (0, gap)
        used += cfg.sk_gap == gap
    assert used > 0


def _brute_force_critical_path(T_sk, KT, G, gap, dp_tiles, store):
    """Longest CTA (k-slices plus `store` per tile stored) when the split tiles'
    slices, each followed by `gap` placeholder positions except the last tile,
    are dealt out to G CTAs as equal ranges of positions.  None: some CTA would
    get no real slice."""
    pos = []
    for t in range(T_sk):
        pos += [t] * KT
        if t < T_sk - 1:
            pos += [None] * gap
    V = len(pos)
    if V // G < gap + 1:
        return None
    worst = 0.0
    for g in range(G):
        real = [t for t in pos[g * V // G:(g + 1) * V // G] if t is not None]
        assert real, "a CTA without a real slice"
        n_dp = len(range(g, dp_tiles, G))
        worst = max(worst, n_dp * (KT + store) + len(real) + len(set(real)) * store)
    return worst


@pytest.mark.parametrize("M,N,K,name,occ", [
    (1024, 1024, 1024, "128x256x32_t8x16_s4_f2_tma", 1),
    (2048, 2048, 2048, "128x256x64_t8x16_s2_f2_v4", 1),
    (4096, 4096, 4096, "128x256x64_t8x16_s2_f2_v4", 1),
    (2048, 2048, 2048, "256x128x64_t8x16_s2_f2_v4", 1),
    (4096, 4096, 4096, "256x128x64_t8x16_s2_f2_v4", 1),
    (8192, 8192, 8192, "256x128x64_t8x16_s2_f2_v4", 1),
    (16384, 64, 4096, "512x64x32_t8x16_s2_f2_v4", 1),
    (1024, 1024, 1024, "256x128x32_t8x16_s4_f2_v4", 1),
    (3001, 2047, 1999, "256x128x32_t8x16_s4_f2_v4", 1),
    (3001, 2047, 1999, "128x256x32_t8x16_s4_f2_tma", 1),
    (16384, 64, 4096, "128x64x16_t16x8_s4_f2_v4", 4),
    (256, 256, 256, "64x64x16_t8x8_s3_f2_v4", 4),
    (1500, 1000, 3000, "128x128x32_t8x8_s3_f2_v4", 2),
    (700, 900, 2500, "128x256x16_t8x16_s6_f2_v4", 1),
])
def test_gap_choice_minimises_the_critical_path(lib, monkeypatch, M, N, K, name, occ):
    """The planner's gap is the smallest one with the shortest longest-CTA time,
    the partition rebuilt here position by position."""
    monkeypatch.delenv("SGEMM_SK_GAP", raising=False)
    monkeypatch.setenv("SGEMM_CLUSTER", "0")
    cfg = _cfg()
    assert lib.sgemm_schedule_check(M, N, K, _kid(lib, name), 152, occ, 0,
                                    ctypes.byref(cfg)) == 0
    KT = -(-K // cfg.bk)
    store = 12.0 / cfg.bk
    dp = cfg.tiles - cfg.sk_tiles
    best, best_cost = 0, None
    if cfg.sk_tiles > 1:
        for gap in range(4):
            c = _brute_force_critical_path(cfg.sk_tiles, KT, cfg.grid, gap, dp, store)
            if c is None:
                break
            if best_cost is None or c < best_cost - 1e-9:
                best, best_cost = gap, c
    assert cfg.sk_gap == best, (cfg.sk_gap, best)


def test_gap_takes_a_store_off_the_1024_cube_critical_path(lib, monkeypatch):
    """1024^3 on 128x256x32 tiles: 32 split tiles of 32 slices over 152 CTAs.  Equal
    ranges give some CTA 7 slices and two partial stores; one placeholder slice per
    boundary leaves 7 slices and one store at most."""
    monkeypatch.delenv("SGEMM_SK_GAP", raising=False)
    cfg = _cfg()
    assert lib.sgemm_schedule_check(1024, 1024, 1024,
                                    _kid(lib, "128x256x32_t8x16_s4_f2_tma"), 152, 1, 0,
                                    ctypes.byref(cfg)) == 0
    assert (cfg.grid, cfg.sk_tiles, cfg.sk_gap) == (152, 32, 1)
    store = 12.0 / 32
    c0 = _brute_force_critical_path(32, 32, 152, 0, 0, store)
    c1 = _brute_force_critical_path(32, 32, 152, 1, 0, store)
    assert c0 == pytest.approx(7 + 2 * store) and c1 == pytest.approx(7 + store)


def test_gap_memo_is_order_independent(lib, monkeypatch):
    """The planner memoises the gap search per thread (16 slots, hashed by the
    schedule's numbers).  Interleaving many schedules, in two orders and with forced
    gaps in between, must give the same gaps as computing each one alone."""
    monkeypatch.delenv("SGEMM_SK_GAP", raising=False)
    n = lib.sgemm_num_kernels()
    cases = [(kid, M, N, K, sms, occ)
             for kid in range(n)
             for (M, N, K) in [(1024, 1024, 1024), (3001, 2047, 1999), (4096, 4096, 4096),
                               (700, 900, 2500), (16384, 64, 4096), (5000, 300, 33)]
             for (sms, occ) in [(152, 1), (148, 2), (13, 4)]]

    def gaps(order):
        out = {}
        for c in order:
            kid, M, N, K, sms, occ = c
            cfg = _cfg()
            assert lib.sgemm_schedule_check(M, N, K, kid, sms, occ, 0, ctypes.byref(cfg)) == 0
            out[c] = cfg.sk_gap
        return out

    first = gaps(cases)
    monkeypatch.setenv("SGEMM_SK_GAP", "2")
    gaps(cases[::3])
    monkeypatch.delenv("SGEMM_SK_GAP")
    assert gaps(cases[::-1]) == first
    assert any(g > 0 for g in first.values()) and any(g == 0 for g in first.values())


# --------------------------------------------------------------------------
# cluster split: each tile's K range cut into S pieces, one per CTA of a
# thread-block cluster, summed in distributed shared memory
# --------------------------------------------------------------------------


def _is_tma(lib, kid):
    return lib.sgemm_kernel_name(kid).decode().endswith("_tma")


def test_cluster_schedule_covers_each_slice_once(lib, monkeypatch):
    """schedule 3: every cp.async entry splits every tile over a cluster whenever
    K has a slice for each CTA; the walk checks each (tile, slice) once, pieces in
    rank order inside tile g / S, and the cluster grid."""
    monkeypatch.delenv("SGEMM_CLUSTER", raising=False)
    n = lib.sgemm_num_kernels()
    seen = set()
    for kid, (M, N, K), (sms, occ) in itertools.product(range(n), SHAPES, MACHINES):
        cfg = _cfg()
        rc = lib.sgemm_schedule_check(M, N, K, kid, sms, occ, 3, ctypes.byref(cfg))
        assert rc == 0, (kid, M, N, K, sms, occ, lib.sgemm_last_error())
        KT = -(-K // cfg.bk)
        if _is_tma(lib, kid):
            assert cfg.cluster == 0
            continue
        want = 1
        while 2 * want <= min(8, KT):
            want *= 2
        assert cfg.cluster == (want if want >= 2 else 0), (kid, M, N, K, cfg.cluster)
        if cfg.cluster:
            assert cfg.grid == cfg.tiles * cfg.cluster and cfg.sk_tiles == cfg.tiles
            assert cfg.split_k == cfg.cluster and cfg.sk_gap == 0
            seen.add(cfg.cluster)
    assert seen == {2, 4, 8}


@pytest.mark.parametrize("S", [2, 4, 8])
def test_forced_cluster_size(lib, monkeypatch, S):
    """SGEMM_CLUSTER=S asks for clusters of up to S CTAs: the largest power of two
    at most S that still gives every CTA a slice (none below 2)."""
    monkeypatch.setenv("SGEMM_CLUSTER", str(S))
    for kid in range(lib.sgemm_num_kernels()):
        for (M, N, K) in [(256, 256, 256), (3001, 2047, 1999), (65, 63, 17), (1, 1, 1)]:
            for schedule in (0, 3):
                cfg = _cfg()
                assert lib.sgemm_schedule_check(M, N, K, kid, 152, 1, schedule,
                                                ctypes.byref(cfg)) == 0
                KT = -(-K // cfg.bk)
                cap = 1
                while 2 * cap <= min(S, KT):
                    cap *= 2
                expect = 0 if _is_tma(lib, kid) or cap < 2 else cap
                if schedule == 0 and expect == 0 and not _is_tma(lib, kid):
                    expect = cfg.cluster   # falls back to the automatic plan
                assert cfg.cluster == expect, (kid, M, N, K, schedule, cfg.cluster)


def test_no_cluster_when_disabled_or_forced_otherwise(lib, monkeypatch):
    monkeypatch.setenv("SGEMM_CLUSTER", "0")
    for kid in range(lib.sgemm_num_kernels()):
        for schedule in (0, 1, 2, 3):
            cfg = _cfg()
            assert lib.sgemm_schedule_check(256, 256, 256, kid, 152, 1, schedule,
                                            ctypes.byref(cfg)) == 0
            assert cfg.cluster == 0
    monkeypatch.delenv("SGEMM_CLUSTER")
    for kid in range(lib.sgemm_num_kernels()):
        for schedule in (1, 2):
            cfg = _cfg()
            assert lib.sgemm_schedule_check(256, 256, 256, kid, 152, 1, schedule,
                                            ctypes.byref(cfg)) == 0
            assert cfg.cluster == 0


def _auto_cluster(T, KT, gmax, occ):
    """The automatic rule, restated: the largest S in 8, 4, 2 with at least 2
    slices per CTA (4 for S = 8) and one resident wave (1.35 for S = 8 when the
    entry keeps 4 or more CTAs per SM); stream-K stays when the cluster grid is
    under 0.9 (one CTA per SM) or 0.6 (several) of stream-K's grid."""
    g_sk = min(max(T * KT // 4, T), gmax)
    for S in (8, 4, 2):
        if KT < S * (4 if S == 8 else 2):
            continue
        if T * S > (1.35 if S == 8 and occ >= 4 else 1.0) * gmax:
            continue
        if T * S < (0.9 if occ == 1 else 0.6) * g_sk:
            return 0
        return S
    return 0


def test_automatic_cluster_rule(lib, monkeypatch):
    """schedule 0 picks a cluster split by the measured rule for problems of less
    than one resident wave of tiles; never for TMA-fed entries."""
    monkeypatch.delenv("SGEMM_CLUSTER", raising=False)
    used = set()
    for kid in range(lib.sgemm_num_kernels()):
        for (M, N, K) in SHAPES + [(128, 128, 128), (384, 384, 384), (512, 512, 512),
                                   (640, 640, 640), (768, 768, 768), (1536, 1536, 1536),
                                   (2048, 256, 256), (4096, 128, 256)]:
            for sms, occ in MACHINES + [(152, 4), (152, 8)]:
                cfg = _cfg()
                assert lib.sgemm_schedule_check(M, N, K, kid, sms, occ, 0,
                                                ctypes.byref(cfg)) == 0
                T, KT, gmax = cfg.tiles, -(-K // cfg.bk), min(sms * occ, 16384)
                expect = 0 if (_is_tma(lib, kid) or T >= gmax) else _auto_cluster(T, KT, gmax,
                                                                                   occ)
                assert cfg.cluster == expect, (kid, M, N, K, sms, occ, cfg.cluster, expect)
                used.add(expect)
    assert used == {0, 2, 4, 8}


@pytest.mark.parametrize("M,N,K,name,occ,S", [
    (128, 128, 128, "32x32x16_t4x4_s3_f2_v4", 8, 4),
    (256, 256, 256, "32x32x16_t4x4_s3_f2_v4", 8, 4),
    (384, 384, 384, "32x32x16_t4x4_s3_f2_v4", 8, 4),
    (512, 512, 512, "64x64x16_t8x8_s3_f2_v4", 4, 8),
    (640, 640, 640, "64x64x16_t8x8_s3_f2_v4", 4, 8),
    (768, 768, 768, "64x64x16_t8x8_s3_f2_v4", 4, 4),
    (1024, 1024, 1024, "256x128x32_t8x16_s4_f2_v4", 1, 0),
    (1536, 1536, 1536, "256x128x32_t8x16_s4_f2_v4", 1, 2),
    (4096, 128, 256, "256x128x64_t8x16_s2_f2_v4", 1, 2),
    (2048, 256, 256, "64x64x16_t8x8_s3_f2_v4", 4, 4),
    (256, 2048, 512, "64x64x16_t8x8_s3_f2_v4", 4, 4),
    (2048, 64, 4096, "64x64x16_t8x8_s3_f2_v4", 4, 0),
    (1024, 64, 4096, "64x64x16_t8x8_s3_f2_v4", 4, 0),
])
def test_measured_cluster_choices(lib, monkeypatch, M, N, K, name, occ, S):
    """The cluster sizes of the timed shapes on 152 SMs."""
    monkeypatch.delenv("SGEMM_CLUSTER", raising=False)
    cfg = _cfg()
    assert lib.sgemm_schedule_check(M, N, K, _kid(lib, name), 152, occ, 0,
                                    ctypes.byref(cfg)) == 0
    assert cfg.cluster == S
