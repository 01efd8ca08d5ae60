// Persistent-grid schedule shared by the kernels and by the host-side checker.
//
// The C tiles are numbered in a grouped raster order.  Tiles [0, dp_tiles) are
// data-parallel: CTA g computes tiles g, g+G, g+2G, ... over their whole K
// range.  The remaining sk_tiles tiles are split by k-slices: their
// sk_iters = sk_tiles * KT slices are cut into G contiguous ranges, one per CTA
// (stream-K).  A CTA walks its data-parallel slices first and then its
// stream-K range as one flat list, so its copy pipeline runs on across tile
// boundaries.
//
// The ranges are equal in a count that may include sk_gap "virtual" slices
// after every split tile but the last.  No CTA computes those; they stand for
// the time a CTA spends storing one more partial tile, so that a range which
// crosses a tile boundary (and ends in two partial-tile stores) holds fewer
// real slices.  sk_gap = 0 gives the plain equal split of sk_iters.
#pragma once

#include <stddef.h>

#include <cmath>

#include "sgemm_args.h"

namespace sgemm {

// ----------------------------------------------------------------------------
// Work schedule of one CTA (persistent grid)
// ----------------------------------------------------------------------------
struct CtaWork {
    int g, G, KT, dp_tiles, n_dp;
    long long u0, u1, dp_iters, total, sk_iters;
};

// Stream-K partition.  Split-tile slice u = t*KT + k sits at virtual position
// v = u + (u / KT) * sk_gap; there are V = sk_iters + (sk_tiles - 1) * sk_gap
// positions, and CTA g owns the real slices with v in [floor(gV/G), floor((g+1)V/G)).
__host__ __device__ __forceinline__ long long sk_virtual_total(const GemmArgs& a) {
    return a.sk_tiles > 0 ? a.sk_iters + static_cast<long long>(a.sk_tiles - 1) * a.sk_gap : 0;
}

// First real slice at or after virtual position v.
__host__ __device__ __forceinline__ long long sk_real_at(long long v, int KT, int gap) {
    const long long P = static_cast<long long>(KT) + gap, t = v / P, k = v - t * P;
    return k >= KT ? (t + 1) * KT : t * KT + k;
}

// The gap > 0 forms of the two lookups below, kept out of line: 64-bit
// divisions are long instruction sequences on the GPU, and with gap 0 the
// kernels' prologue then carries only the equal split's one.
inline __host__ __device__ __noinline__ long long sk_begin_gap(const GemmArgs& a, int g) {
    return sk_real_at(sk_virtual_total(a) * g / a.grid, a.KT, a.sk_gap);
}
inline __host__ __device__ __noinline__ int sk_owner_gap(const GemmArgs& a, long long u) {
    const long long v = u + (u / a.KT) * a.sk_gap;
    return static_cast<int>(((v + 1) * a.grid - 1) / sk_virtual_total(a));
}

// First slice of CTA g's stream-K range; g = G gives sk_iters.
__host__ __device__ __forceinline__ long long sk_begin(const GemmArgs& a, int g) {
    return a.sk_gap == 0 ? a.sk_iters * g / a.grid : sk_begin_gap(a, g);
}

// The CTA whose range holds slice u: the g with floor(gV/G) <= v < floor((g+1)V/G),
// which is floor(((v + 1) G - 1) / V).
__host__ __device__ __forceinline__ int sk_owner(const GemmArgs& a, long long u) {
    return a.sk_gap == 0 ? static_cast<int>(((u + 1) * a.grid - 1) / a.sk_iters)
                         : sk_owner_gap(a, u);
}

__host__ __device__ __forceinline__ CtaWork make_work(const GemmArgs& a, int g) {
    CtaWork w;
    w.g = g;
    w.G = a.grid;
    w.KT = a.KT;
    w.dp_tiles = a.dp_tiles;
    w.n_dp = (w.g < a.dp_tiles) ? (a.dp_tiles - 1 - w.g) / w.G + 1 : 0;
    w.sk_iters = a.sk_iters;
    w.u0 = sk_begin(a, w.g);       // 0 when no tile is split (sk_iters = 0, gap 0)
    w.u1 = sk_begin(a, w.g + 1);
    w.dp_iters = static_cast<long long>(w.n_dp) * w.KT;
    w.total = w.dp_iters + (w.u1 - w.u0);
    return w;
}

// make_work for a cluster split (a.cl_split = S, a power of two): CTA g = t*S + r
// holds slices [floor(KT*r/S), floor(KT*(r+1)/S)) of tile t, which is what
// make_work gives for G = T*S and no data-parallel tiles, with shifts in place
// of its 64-bit divisions (the host-side schedule check compares the two).
__host__ __device__ __forceinline__ CtaWork make_cluster_work(const GemmArgs& a, int g) {
    int sh = 0;
    while ((1 << sh) < a.cl_split) ++sh;
    const long long t = g >> sh, r = g & (a.cl_split - 1);
    const long long tb = t * a.KT;
    CtaWork w;
    w.g = g;
    w.G = a.grid;
    w.KT = a.KT;
    w.dp_tiles = 0;
    w.n_dp = 0;
    w.sk_iters = a.sk_iters;
    w.u0 = tb + ((a.KT * r) >> sh);
    w.u1 = tb + ((a.KT * (r + 1)) >> sh);
    w.dp_iters = 0;
    w.total = w.u1 - w.u0;
    return w;
}

// Partial-tile slot (0 or 1) CTA w uses for split tile t: a CTA's stream-K range
// is shorter than one tile's K range plus one gap, so it touches at most two
// split tiles.
__host__ __device__ __forceinline__ int sk_slot(const CtaWork& w, int t) {
    return t - static_cast<int>(w.u0 / w.KT);
}

// Position in the CTA's flat list of k-slices.
struct Cursor {
    long long c;
    int tile, kt, kt_begin, kt_end;

    __host__ __device__ __forceinline__ void seek(const CtaWork& w, long long c_) {
        c = c_;
        if (c < w.dp_iters) {
            const int j = static_cast<int>(c / w.KT);
            tile = w.g + j * w.G;
            kt = static_cast<int>(c - static_cast<long long>(j) * w.KT);
            kt_begin = 0;
            kt_end = w.KT;
        } else {
            const long long u = w.u0 + (c - w.dp_iters);
            const int t = static_cast<int>(u / w.KT);
            const long long tb = static_cast<long long>(t) * w.KT;
            tile = w.dp_tiles + t;
            kt = static_cast<int>(u - tb);
            kt_begin = static_cast<int>((w.u0 > tb ? w.u0 : tb) - tb);
            const long long te = tb + w.KT;
            kt_end = static_cast<int>((w.u1 < te ? w.u1 : te) - tb);
        }
    }
    // Piece [kb, ke) of tile `t` as the whole list (a cluster-split CTA).
    __host__ __device__ __forceinline__ void set_piece(int t, int kb, int ke) {
        c = 0;
        tile = t;
        kt = kt_begin = kb;
        kt_end = ke;
    }
    __host__ __device__ __forceinline__ void advance(const CtaWork& w) {
        ++c;
        ++kt;
        if (kt >= kt_end && c < w.total) seek(w, c);
    }
};

// Tile index -> origin of the tile in C.  Tiles are rasterised in groups of
// group_m tile rows so that CTAs running together share A and B panels in L2.
__host__ __device__ __forceinline__ void tile_origin(const GemmArgs& a, int tile, int BM,
                                                     int BN, int& m0, int& n0) {
    const int group_size = a.group_m * a.tiles_n;
    const int group = tile / group_size;
    const int first_m = group * a.group_m;
    const int rows = (a.tiles_m - first_m < a.group_m) ? a.tiles_m - first_m : a.group_m;
    const int r = tile - group * group_size;
    m0 = (first_m + r % rows) * BM;
    n0 = (r / rows) * BN;
}

// ----------------------------------------------------------------------------
// Host-side planning of the schedule above
// ----------------------------------------------------------------------------
constexpr int kMinSkIters = 4;   // fewest k-slices a CTA gets when all tiles are split
constexpr size_t kWsAlign = 256;
constexpr int kMaxSkTiles = 16384;   // ceiling on the persistent grid
constexpr int kMaxSplit = 256;       // most CTAs that may share one split tile

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SchedSizes {
    int split = 1;              // most CTAs sharing one split tile
    size_t partial_bytes = 0;   // workspace bytes of partial tiles
};

constexpr int kMaxSkGap = 3;   // largest gap the automatic choice tries

// Longest CTA of the current schedule, in k-slices, when storing a tile (whole
// or partial) costs `store` slices: the quantity the gap choice minimises.
inline double sk_critical_path(const GemmArgs& a, double store) {
    double worst = 0.0;
    const int extra = a.dp_tiles % a.grid;   // CTAs [0, extra) hold one more whole tile
    const int n_dp_lo = a.dp_tiles / a.grid;
    long long u0 = sk_begin(a, 0);
    for (int g = 0; g < a.grid; ++g) {
        const long long u1 = sk_begin(a, g + 1);
        const int n_dp = n_dp_lo + (g < extra ? 1 : 0);
        const long long pieces = u1 > u0 ? (u1 - 1) / a.KT - u0 / a.KT + 1 : 0;
        const double c = n_dp * (a.KT + store) + static_cast<double>(u1 - u0) + pieces * store;
        if (c > worst) worst = c;
        u0 = u1;
    }
    return worst;
}

// Gap for the stream-K partition (see the top of this file): the smallest one in
// [0, kMaxSkGap] with the shortest critical path, among those that leave every
// CTA at least one real slice.  forced >= 0 asks for that gap, if it is allowed.
inline int choose_sk_gap(GemmArgs& a, double store, int forced) {
    if (a.sk_tiles <= 1) return 0;
    // The search walks every CTA for each gap (microseconds of host time per
    // call); its answer depends on these few numbers only, so each thread keeps
    // the last answers for a handful of schedules.
    struct Memo {
        long long sk_iters;
        int sk_tiles, KT, grid, dp_tiles, forced, gap;
        double store;
        bool used;
    };
    static thread_local Memo memo[16];
    const unsigned slot = (static_cast<unsigned>(a.sk_tiles) * 2654435761u ^
                           static_cast<unsigned>(a.KT) * 40503u ^
                           static_cast<unsigned>(a.grid) * 97u ^
                           static_cast<unsigned>(a.dp_tiles) * 13u) % 16u;
    Memo& m = memo[slot];
    if (m.used && m.sk_iters == a.sk_iters && m.sk_tiles == a.sk_tiles && m.KT == a.KT &&
        m.grid == a.grid && m.dp_tiles == a.dp_tiles && m.forced == forced && m.store == store)
        return m.gap;
    int best = 0;
    double best_cost = 0.0;
    for (int gap = 0; gap <= (forced >= 0 ? forced : kMaxSkGap); ++gap) {
        a.sk_gap = gap;
        // Ranges of at least gap + 1 positions always hold a real slice.
        if (sk_virtual_total(a) / a.grid < gap + 1) break;
        if (forced >= 0) {
            if (gap == forced) best = gap;
            continue;
        }
        const double c = sk_critical_path(a, store);
        if (gap == 0 || c < best_cost - 1e-9) {
            best = gap;
            best_cost = c;
        }
    }
    m = Memo{a.sk_iters, a.sk_tiles, a.KT, a.grid, a.dp_tiles, forced, best, store, true};
    return best;
}

// Cluster split (cl_split = S > 1).  Every tile's K range is cut into S
// contiguous pieces, one per CTA, and the S CTAs of a tile are one thread-block
// cluster: CTAs t*S .. t*S+S-1 hold tile t, rank r holding the r-th piece.  It is
// the stream-K partition above with G = T*S, no data-parallel tiles and no gap,
// which gives CTA t*S+r the slices [floor(KT*r/S), floor(KT*(r+1)/S)) of tile t.
// The partials are summed inside the cluster in rank (= k) order, so no
// workspace and no second launch are needed.
constexpr int kMaxCluster = 8;        // portable cluster size
constexpr int kMaxClusterGrid = 1 << 22;

// Automatic cluster size for T tiles of KT slices on a resident grid of gmax
// CTAs (occ per SM), 0 for none.  Chosen from CUDA-event step times on GB300
// (L2 flushed before each step; 128^3 .. 1536^3 cubes and narrow shapes such as
// 2048x256x256 and 4096x128x256), where the rule below picked the fastest of
// S = 0, 2, 4, 8 or came within 5 % of it:
//   * at least 2 slices per CTA, and 4 for clusters of 8 (one- and two-slice
//     pieces in clusters of 8 lost to clusters of 4 at 128^3 .. 384^3);
//   * one resident wave (T*S <= gmax); clusters of 8 of an entry with 4 or more
//     CTAs per SM may take up to 1.35 waves (640^3 on 64 x 64 tiles);
//   * stream-K stays when the cluster grid is well below stream-K's own grid:
//     under 0.9 of it for an entry with one CTA per SM (1024^3 on 256 x 128
//     tiles: 128 clustered CTAs ran 53.6 us, 152 stream-K CTAs 51.5 us), under 0.6
//     for entries with several (2048 x 64 x 4096 on 64 x 64 tiles: 256 clustered
//     CTAs 41.0 us, 608 stream-K CTAs 35.7; 384^3 at 0.67 and 256 x 2048 x 512 at
//     0.84 of it still ran 9 % faster clustered).
inline int auto_cluster_size(long long T, int KT, long long gmax, int occ, int cap) {
    long long g_sk = T * KT / kMinSkIters;   // stream-K's grid for the same tiles
    if (g_sk < T) g_sk = T;
    if (g_sk > gmax) g_sk = gmax;
    const double keep_sk_below = occ == 1 ? 0.9 : 0.6;
    for (int S = cap; S >= 2; S /= 2) {
        const int min_slices = S >= 8 ? 4 : 2;
        if (KT < static_cast<long long>(S) * min_slices) continue;
        const double waves = (S >= 8 && occ >= 4) ? 1.35 : 1.0;
        if (static_cast<double>(T * S) > waves * static_cast<double>(gmax)) continue;
        if (static_cast<double>(T * S) < keep_sk_below * static_cast<double>(g_sk)) return 0;
        return S;
    }
    return 0;
}

// Cluster size for T tiles of KT slices: the largest power of two S <= cap with
// at least min_slices slices per CTA and T*S <= gmax (0 when below 2).
inline int cluster_size_for(long long T, int KT, long long gmax, int cap, int min_slices) {
    int s = 1;
    while (2 * s <= cap && static_cast<long long>(KT) >= 2LL * s * min_slices &&
           T * 2 * s <= gmax)
        s *= 2;
    return s >= 2 ? s : 0;
}

// Fills the schedule fields of `a` (a.M, a.N, a.K set) for BM x BN x BK tiles on
// `sms` SMs holding `occ` CTAs each.  schedule: 0 automatic, 1 data-parallel
// only, 2 stream-K on any partial wave that has at least one k-slice per CTA,
// 3 cluster split of every tile (see above) wherever K has a slice per CTA.
// store_slices: cost of storing one tile in k-slices (0: equal stream-K ranges,
// no gap); forced_gap >= 0 overrides the gap choice where it is allowed;
// group_m > 0 sets the raster group height (0: chosen from the tile shape).
// cluster_max: largest cluster the kernel can sum in (0: none); forced_cluster:
// -1 automatic, 0 never, S >= 2 clusters of the largest power of two up to S
// that gives every CTA a slice.
inline SchedSizes plan_schedule(GemmArgs& a, int bm, int bn, int bk, int sms, int occ,
                                int schedule, double store_slices = 0.0,
                                int forced_gap = -1, int group_m = 0, int cluster_max = 0,
                                int forced_cluster = -1) {
    a.tiles_m = (a.M + bm - 1) / bm;
    a.tiles_n = (a.N + bn - 1) / bn;
    a.KT = (a.K + bk - 1) / bk;
    a.cl_split = 0;
    const long long T = static_cast<long long>(a.tiles_m) * a.tiles_n;
    long long Gmax = static_cast<long long>(sms) * occ;
    if (Gmax > kMaxSkTiles) Gmax = kMaxSkTiles;
    // Raster groups of group_m tile rows.  A wave of G tiles spanning r tile rows
    // and G/r columns reads r*BM rows of A and (G/r)*BN columns of B per k; that
    // is least for r = sqrt(G*BN/BM).  group_m is the power of two nearest to it
    // (16 for 128 x 256 tiles on 152 SMs, 8 for 256 x 128), so waves repeat
    // fewer DRAM reads of either operand.
    if (group_m <= 0) {
        const double r = std::sqrt(static_cast<double>(Gmax) * bn / bm);
        group_m = 1;
        while (group_m < 4096 && group_m * 1.4142135623730951 < r) group_m *= 2;
    }
    a.group_m = a.tiles_m < group_m ? a.tiles_m : group_m;

    // Cluster split: forced (schedule 3 or a forced size), or automatic for
    // problems of less than one resident wave of tiles (auto_cluster_size).
    if (cluster_max >= 2 && schedule != 1 && schedule != 2 && forced_cluster != 0) {
        const int cap = cluster_max < kMaxCluster ? cluster_max : kMaxCluster;
        int S = 0;
        if (forced_cluster >= 2 || schedule == 3) {
            const int want = forced_cluster >= 2 ? forced_cluster : cap;
            S = cluster_size_for(T, a.KT, kMaxClusterGrid, want < cap ? want : cap, 1);
        } else if (T < Gmax) {
            S = auto_cluster_size(T, a.KT, Gmax, occ, cap);
        }
        if (S >= 2) {
            a.grid = static_cast<int>(T * S);
            a.dp_tiles = 0;
            a.sk_tiles = static_cast<int>(T);
            a.sk_iters = T * a.KT;
            a.sk_gap = 0;
            a.cl_split = S;
            SchedSizes z;
            z.split = S;
            return z;
        }
    }

    long long G, dp, sk;
    if (T >= Gmax) {
        // Whole waves run data-parallel; a partial last wave is shared out by
        // k-slices when every CTA gets at least one and the shared tail (its
        // slices plus about two slices of partial stores and reduction) is
        // shorter than the extra wave of whole tiles it replaces: 4096 x 4096 x
        // 512 on 128 x 256 x 64 tiles, 56 tiles of 8 slices past 3 waves, ran
        // 52.7 TFLOP/s with the extra wave, where its 32-deep twin, whose 16
        // slices a tile let stream-K take those tiles, ran 57.3.
        G = Gmax;
        const long long rem = T % Gmax;
        const long long tail = (rem * a.KT + Gmax - 1) / Gmax;   // slices per CTA
        const bool use_sk = rem != 0 && schedule != 1 && rem * a.KT >= Gmax &&
                            (schedule == 2 || tail + 2 < a.KT);
        sk = use_sk ? rem : 0;
        dp = T - sk;
    } else {
        // Fewer tiles than resident CTAs: split every tile's K range over more CTAs.
        long long want = (schedule == 1) ? T : T * a.KT / kMinSkIters;
        if (schedule == 2) want = T * a.KT;
        if (want > Gmax) want = Gmax;
        if (want > T) {
            G = want;
            dp = 0;
            sk = T;
        } else {
            G = T;
            dp = T;
            sk = 0;
        }
    }
    SchedSizes z;
    for (;;) {
        a.grid = static_cast<int>(G);
        a.dp_tiles = static_cast<int>(dp);
        a.sk_tiles = static_cast<int>(sk);
        a.sk_iters = sk * a.KT;
        a.sk_gap = 0;
        if (store_slices > 0.0 || forced_gap >= 0)
            a.sk_gap = choose_sk_gap(a, store_slices, forced_gap);
        z.split = 1;
        for (long long t = 0; t < sk; ++t) {
            const long long tb = t * a.KT, te = tb + a.KT - 1;
            const int g0 = sk_owner(a, tb);
            const int g1 = sk_owner(a, te);
            if (g1 - g0 + 1 > z.split) z.split = g1 - g0 + 1;
        }
        // The reduction handles at most kMaxSplit contributors per tile: use fewer
        // CTAs (or none) for the split tiles otherwise.
        if (z.split <= kMaxSplit) break;
        if (dp == 0 && G / 2 > T) {
            G /= 2;
        } else {
            G = dp > 0 ? G : T;
            dp = T;
            sk = 0;
        }
    }
    if (sk > 0) z.partial_bytes = align_up(static_cast<size_t>(G) * 2 * bm * bn * 4, kWsAlign);
    return z;
}

}  // namespace sgemm
