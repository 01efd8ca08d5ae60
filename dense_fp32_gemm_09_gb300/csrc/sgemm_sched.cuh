// Persistent-grid schedule shared by the kernels and by the host-side checker.
//
// The C tiles are numbered in a grouped raster order.  Tiles [0, dp_tiles) are
// data-parallel: CTA g computes tiles g, g+G, g+2G, ... over their whole K
// range.  The remaining sk_tiles tiles are split by k-slices: their
// sk_iters = sk_tiles * KT slices are cut into G contiguous ranges
// [floor(g*I/G), floor((g+1)*I/G)), one per CTA (stream-K).  A CTA walks its
// data-parallel slices first and then its stream-K range as one flat list, so
// its copy pipeline runs on across tile boundaries.
#pragma once

#include <stddef.h>

#include "sgemm_args.h"

namespace sgemm {

// ----------------------------------------------------------------------------
// Work schedule of one CTA (persistent grid)
// ----------------------------------------------------------------------------
struct CtaWork {
    int g, G, KT, dp_tiles, n_dp;
    long long u0, u1, dp_iters, total, sk_iters;
};

__host__ __device__ __forceinline__ CtaWork make_work(const GemmArgs& a, int g) {
    CtaWork w;
    w.g = g;
    w.G = a.grid;
    w.KT = a.KT;
    w.dp_tiles = a.dp_tiles;
    w.n_dp = (w.g < a.dp_tiles) ? (a.dp_tiles - 1 - w.g) / w.G + 1 : 0;
    w.sk_iters = a.sk_iters;
    w.u0 = a.sk_iters * w.g / w.G;
    w.u1 = a.sk_iters * (w.g + 1) / w.G;
    w.dp_iters = static_cast<long long>(w.n_dp) * w.KT;
    w.total = w.dp_iters + (w.u1 - w.u0);
    return w;
}

// The CTA whose stream-K range holds shared k-slice u:
// ranges are [floor(g*I/G), floor((g+1)*I/G)), so it is floor(((u+1)G - 1) / I).
__host__ __device__ __forceinline__ int sk_owner(long long u, int G, long long I) {
    return static_cast<int>(((u + 1) * G - 1) / I);
}

// Partial-tile slot (0 or 1) CTA w uses for split tile t: a CTA's stream-K range
// is shorter than one tile's K range, so it touches at most two split tiles.
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
    __host__ __device__ __forceinline__ void advance(const CtaWork& w) {
        ++c;
        ++kt;
        if (kt >= kt_end) seek(w, c);
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
constexpr int kMinSkIters = 4;   // fewest k-slices a CTA gets when tiles are split
constexpr size_t kWsAlign = 256;
constexpr int kMaxSkTiles = 16384;   // ceiling on the persistent grid
constexpr int kMaxSplit = 256;       // most CTAs that may share one split tile

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SchedSizes {
    int split = 1;              // most CTAs sharing one split tile
    size_t partial_bytes = 0;   // workspace bytes of partial tiles
};

// Fills the schedule fields of `a` (a.M, a.N, a.K set) for BM x BN x BK tiles on
// `sms` SMs holding `occ` CTAs each.  schedule: 0 automatic, 1 data-parallel
// only, 2 stream-K on any partial wave that has at least one k-slice per CTA.
inline SchedSizes plan_schedule(GemmArgs& a, int bm, int bn, int bk, int sms, int occ,
                                int schedule) {
    a.tiles_m = (a.M + bm - 1) / bm;
    a.tiles_n = (a.N + bn - 1) / bn;
    a.KT = (a.K + bk - 1) / bk;
    // 16 tile rows per raster group: a wave of ~152 tiles then spans about 16 rows
    // x 9.5 columns rather than 8 rows x all columns, so each wave reads A rows
    // and B columns in a ratio near the optimum (fewer repeated B reads from DRAM).
    a.group_m = a.tiles_m < 16 ? a.tiles_m : 16;
    const long long T = static_cast<long long>(a.tiles_m) * a.tiles_n;
    long long Gmax = static_cast<long long>(sms) * occ;
    if (Gmax > kMaxSkTiles) Gmax = kMaxSkTiles;

    long long G, dp, sk;
    if (T >= Gmax) {
        // Whole waves run data-parallel; a partial last wave is shared out by
        // k-slices when every CTA gets enough of them.
        G = Gmax;
        const long long rem = T % Gmax;
        const bool use_sk = rem != 0 && schedule != 1 &&
                            (schedule == 2 ? rem * a.KT >= Gmax
                                           : rem * a.KT >= Gmax * kMinSkIters);
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
        z.split = 1;
        for (long long t = 0; t < sk; ++t) {
            const long long tb = t * a.KT, te = tb + a.KT - 1;
            const int g0 = sk_owner(tb, static_cast<int>(G), a.sk_iters);
            const int g1 = sk_owner(te, static_cast<int>(G), a.sk_iters);
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
