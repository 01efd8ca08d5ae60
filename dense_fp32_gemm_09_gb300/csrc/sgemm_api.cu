// Host side of the C ABI declared in include/sgemm.h: argument checks, the
// tile table and its selection, the persistent / stream-K schedule, workspaces
// and launches.  No torch type crosses this boundary.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "sgemm_ffma_tma.cuh"
#include "sgemm_internal.h"
#include "sgemm_sched.cuh"
#include "sgemm_tma_host.h"

namespace sgemm {

const KernelEntry* ffma_entries_main(int* count);
const KernelEntry* ffma_entries_small(int* count);
const KernelEntry* ffma_entries_any(int* count);
const KernelEntry* ffma_entries_tma(int* count);

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char t_last_error[512] = "";

void set_error(const char* what, cudaError_t e) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%s)", what,
                  cudaGetErrorName(e), cudaGetErrorString(e));
}

// ----------------------------------------------------------------------------
// Tile table
// ----------------------------------------------------------------------------
const std::vector<KernelEntry>& table() {
    static const std::vector<KernelEntry> t = [] {
        std::vector<KernelEntry> v;
        int n = 0;
        const KernelEntry* e = ffma_entries_main(&n);
        v.insert(v.end(), e, e + n);
        e = ffma_entries_small(&n);
        v.insert(v.end(), e, e + n);
        e = ffma_entries_any(&n);
        v.insert(v.end(), e, e + n);
        e = ffma_entries_tma(&n);
        v.insert(v.end(), e, e + n);
        return v;
    }();
    return t;
}

int find_entry(const char* name) {
    const auto& t = table();
    for (size_t i = 0; i < t.size(); ++i)
        if (std::strcmp(t[i].name, name) == 0) return static_cast<int>(i);
    return -1;
}

// Per-device facts and per-(device, entry) residency, computed once per device
// (and again after sgemm_shutdown), with each kernel's shared-memory attributes
// set in the device's context on the way.
struct DeviceInfo {
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    std::vector<int> occ;  // resident CTAs per SM for each table entry (0 = unusable)
    // Clusters of 2, 4 and 8 CTAs of each entry that can be resident at once
    // (cudaOccupancyMaxActiveClusters).  A cluster must sit inside one GPC, so at
    // one CTA per SM only 15 clusters of 8 fit on 152 SMs, not 19.
    std::vector<std::array<int, 3>> clusters;
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

int device_info(int dev, const DeviceInfo** out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
        *out = &it->second;
        return SGEMM_OK;
    }
    DeviceInfo info;
    cudaError_t e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) {
        set_error("cudaDeviceGetAttribute", e);
        return SGEMM_ERR_LAUNCH;
    }
    if (info.cc_major != 10 || info.cc_minor != 3) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                      info.cc_major, info.cc_minor);
        return SGEMM_ERR_UNSUPPORTED;
    }
    const auto& t = table();
    info.occ.assign(t.size(), 0);
    info.clusters.assign(t.size(), {0, 0, 0});
    for (size_t i = 0; i < t.size(); ++i) {
        e = cudaFuncSetAttribute(t[i].kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 t[i].smem_bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(t[i].kernel,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        int occ = 0;
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, t[i].kernel, t[i].threads,
                                                              t[i].smem_bytes);
        if (e != cudaSuccess) {
            set_error("kernel attribute / occupancy query", e);
            return SGEMM_ERR_LAUNCH;
        }
        info.occ[i] = occ;
        info.clusters[i] = {0, 0, 0};
        if (t[i].tma || occ <= 0) continue;   // only the cp.async kernels sum in clusters
        for (int l = 0; l < 3; ++l) {
            const unsigned S = 2u << l;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = S;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cudaLaunchConfig_t c{};
            c.gridDim = dim3(S);
            c.blockDim = dim3(static_cast<unsigned>(t[i].threads));
            c.dynamicSmemBytes = static_cast<size_t>(t[i].smem_bytes);
            c.attrs = at;
            c.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, t[i].kernel, &c) != cudaSuccess) {
                cudaGetLastError();   // a size the kernel cannot take: never chosen
                n = 0;
            }
            info.clusters[i][l] = n;
        }
    }
    auto res = g_dev.emplace(dev, std::move(info));
    *out = &res.first->second;
    return SGEMM_OK;
}

// ----------------------------------------------------------------------------
// Argument checks
// ----------------------------------------------------------------------------
bool ranges_overlap(const float* p, long long n, const float* q, long long m) {
    if (n <= 0 || m <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), a1 = a0 + 4ull * n;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(q), b1 = b0 + 4ull * m;
    return a0 < b1 && b0 < a1;
}

// Elements spanned by a rows x cols row-major matrix with leading dimension ld.
long long span(int rows, int cols, int ld) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<long long>(rows - 1) * ld + cols;
}

// Tile and slice bounds (m0 + BM, k0 + BK, ...) are 32-bit in the kernels and the
// schedule; element offsets are 64-bit.  Dimensions up to 2^30 keep every such
// bound far from overflow (an fp32 matrix with 2^30 rows of one column is already
// 4 GiB), so larger ones are refused before anything is planned.
constexpr int kMaxDim = 1 << 30;

int check_dims(int M, int N, int K) {
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "dimension above 2^30: M=%d N=%d K=%d", M, N, K);
        return SGEMM_ERR_UNSUPPORTED;
    }
    return SGEMM_OK;
}

// Argument checks for C[M x N] = op(A)[M x K] . op(B)[K x N]: op(A) = A stored
// M x K (transa == 0) or A^T with A stored K x M (transa == 1); likewise B.
int check_args_op(int transa, int transb, int M, int N, int K, const float* A, int lda,
                  const float* B, int ldb, const float* C, int ldc) {
    if (M < 0 || N < 0 || K < 0) {
        std::snprintf(t_last_error, sizeof(t_last_error), "negative size M=%d N=%d K=%d", M,
                      N, K);
        return SGEMM_ERR_INVALID_ARG;
    }
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    const int ra = transa ? K : M, ca = transa ? M : K;   // stored A: ra x ca
    const int rb = transb ? N : K, cb = transb ? K : N;   // stored B: rb x cb
    if (lda < std::max(ca, 1) || ldb < std::max(cb, 1) || ldc < std::max(N, 1)) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "leading dimension below row width: lda=%d (needs %d) ldb=%d (needs %d) "
                      "ldc=%d (N=%d)",
                      lda, ca, ldb, cb, ldc, N);
        return SGEMM_ERR_INVALID_ARG;
    }
    if ((M > 0 && N > 0 && C == nullptr) || (M > 0 && N > 0 && K > 0 && (A == nullptr ||
                                                                          B == nullptr))) {
        std::snprintf(t_last_error, sizeof(t_last_error), "null pointer with non-empty extent");
        return SGEMM_ERR_INVALID_ARG;
    }
    if (M > 0 && N > 0 && K > 0) {
        const long long sc = span(M, N, ldc);
        if (ranges_overlap(C, sc, A, span(ra, ca, lda)) ||
            ranges_overlap(C, sc, B, span(rb, cb, ldb))) {
            std::snprintf(t_last_error, sizeof(t_last_error), "C overlaps A or B");
            return SGEMM_ERR_INVALID_ARG;
        }
    }
    return SGEMM_OK;
}

int check_args(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
               const float* C, int ldc) {
    return check_args_op(0, 0, M, N, K, A, lda, B, ldb, C, ldc);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------------------------
// Selection and schedule
// ----------------------------------------------------------------------------
struct Plan {
    int entry = -1;
    GemmArgs args{};
    size_t ws_partial_bytes = 0;  // bytes of partial tiles
    int ctas_per_sm = 0;
    int split = 1;
    int sms = 0;
};


// 16-byte cp.async needs every A and B row to start on a 16-byte boundary.
bool vec4_ok(const float* A, int lda, const float* B, int ldb) {
    return aligned16(A) && aligned16(B) && (lda % 4 == 0) && (ldb % 4 == 0);
}

bool entry_fits(const KernelEntry& e, const float* A, int lda, const float* B, int ldb) {
    return e.vec != 4 || vec4_ok(A, lda, B, ldb);
}

// The per-shape rules on their own: `sms` SMs, `v4` when 16-byte loads serve A and B.
int choose_by_rules(int sms, int M, int N, int K, bool v4) {
    const long long tiles128 = static_cast<long long>((M + 127) / 128) * ((N + 127) / 128);
    const long long tiles64 = static_cast<long long>((M + 63) / 64) * ((N + 63) / 64);
    const char* name;
    if (v4 && N <= 64 && M >= 2560)
        // Narrow C: 512-row tiles once M fills 5 of them (3000 x 64 x 3000: 25.2
        // TFLOP/s against 22.2 on 64 x 64 tiles; at 2048 x 64 x 4096 the 64 x 64
        // tiles were ahead, 27.8 against 27.1).
        name = "512x64x32_t8x16_s2_f2_v4";
    else if (v4 && tiles64 * 4 <= sms && K <= 1024)
        // The smallest problems: 32 x 32 tiles give the SMs four times as many
        // tiles (256^3: 10.9 against 13.0 us; 384^3: 13.0-14.0 against 15.0).
        name = "32x32x16_t4x4_s3_f2_v4";
    else if (v4 && N <= 64)
        name = "64x64x16_t8x8_s3_f2_v4";
    else if (v4 && M <= 64)
        // Short, wide C: tiles no taller than C (64 x 8192 x 4096: 37.2 TFLOP/s on
        // 64 x 64 tiles against 14.5 on 256 x 128; 32 x 16384 x 4096: 24.6 on 32 x 32
        // against 7.5).
        name = M <= 32 ? "32x32x16_t4x4_s3_f2_v4" : "64x64x16_t8x8_s3_f2_v4";
    else if (v4 && M >= 4096 && N <= 256 && (N + 63) / 64 * 64 < (N + 127) / 128 * 128)
        // Narrow C whose width 64-wide tiles fit more closely than 128-wide ones
        // (8192 x 192 x 4096: 55.5 on 512 x 64 tiles against 43.3 on 256 x 128).
        name = "512x64x32_t8x16_s2_f2_v4";
    else if (v4 && N <= 128 && M >= 4096) {
        // A 256-wide tile would compute half its columns for nothing.  How deep the
        // slices of the 256 x 128 tiles can be depends on how many there are to
        // share out: 64-deep from 4 a CTA (8192 x 128 x 8192, 4096 x 96 x 4096),
        // 32-deep from 1.25 (4096 x 128 x 1024: 32.1 TFLOP/s against 20.7 for
        // 64-deep; 8192 x 128 x 1024: 41.4 against 39.9), else 128 x 128 tiles
        // (4096 x 128 x 512: 23.2 against 16.1).
        const long long slices_h =
            static_cast<long long>((M + 255) / 256) * ((N + 127) / 128) * ((K + 63) / 64);
        name = slices_h >= 4LL * sms ? "256x128x64_t8x16_s2_f2_v4"
             : 4 * slices_h >= 5LL * sms ? "256x128x32_t8x16_s4_f2_v4"
                                         : "128x128x32_t8x8_s3_f2_v4";
    }
    else if (!v4 && M > 64 && N > 64 && tiles128 >= 32 && tiles128 < 128)
        // 4-byte loads, between 32 and 128 tiles of 128 x 128: the 16 x 8 register
        // tile on them (1000 x 1000 x 300: 19.1 TFLOP/s against 16.0 on 128 x 256;
        // 700 x 700 x 1000: 21.5 against 19.7 on 64 x 64).
        name = "128x128x16_t16x8_s4_f2_v1";
    else if (tiles128 * 4 < sms) {
        // Small C.  With K >= 2048 every tile's long K range is shared out (stream-K
        // or a cluster split), and larger register tiles beat 64 x 64 ones where
        // they cover C closely: 128 x 256 tiles from 8 of them with at most a
        // quarter of their area to spare, or from 4 with at most a tenth (768 x 768
        // x 4096: 49.9 against 41.9 TFLOP/s; 512 x 512 x 8192: 50.8 against 37.2;
        // 448 x 448 x 4096: 31.7 against 27.4; 256 x 512 x 8192: 43.1 against
        // 37.7), else 128 x 128 tiles from 9 with at most a fifth to spare (384 x
        // 384 x 2048: 26.0 against 22.1, where the six 128 x 256 tiles, a quarter
        // empty, fall behind both).  320 x 320 x 4096, whose larger tiles would be a
        // third empty, stays on 64 x 64 tiles (25.1 against 22.4).
        // With N <= 128 the 256 x 128 orientation of the same tile fits C's width
        // (2048 x 128 x 2048: 32.1 against 30.3 on 128 x 128 tiles).
        const bool tall = N <= 128;
        const long long tiles_w = tall
            ? static_cast<long long>((M + 255) / 256) * ((N + 127) / 128)
            : static_cast<long long>((M + 127) / 128) * ((N + 255) / 256);
        const double area = static_cast<double>(M) * N;
        const bool wide_ok = tiles_w >= 4 && area >= (tiles_w >= 8 ? 0.75 : 0.9) * tiles_w *
                                                         (128.0 * 256.0);
        const bool quad_ok = tiles128 >= 9 && area >= 0.8 * tiles128 * (128.0 * 128.0);
        if (v4 && K >= 2048 && (wide_ok || quad_ok))
            name = wide_ok ? (tall ? "256x128x32_t8x16_s4_f2_v4" : "128x256x32_t8x16_s4_f2_v4")
                           : "128x128x32_t8x8_s3_f2_v4";
        else
            name = v4 ? "64x64x16_t8x8_s3_f2_v4" : "64x64x16_t8x8_s3_f2_v1";
    } else if (v4) {
        // 64-deep slices run about 3% faster; 32-deep ones share K out more finely
        // over the stream-K ranges.  The deeper ones win once every CTA gets about
        // 16 of them, whatever K (1536^3, 11 a CTA, loses; 2048^3, 27, wins; with
        // K = 2048 but 5 a CTA, 896 x 768 x 2048 ran 35.9 TFLOP/s on 64-deep slices
        // against 43.9 on 32-deep ones, 768 x 1024 x 2048 42.1 against 44.5).
        // Among the 64-deep entries the one with double-buffered fragments (128 x
        // 256) wins once every CTA gets about 44 of its slices (4096^3 65.9 against
        // 64.4 TFLOP/s, 8192^3 67.1 against 65.2, 3072^3 64.1 against 63.2,
        // 4096 x 4096 x 1024 62.5 against 61.8, 8192 x 8192 x 512 63.0 against
        // 62.0); with fewer the 256 x 128 entry does (2048^3 59.4 against 58.9,
        // 2560 x 2560 x 1280 58.4 against 57.2, 3008 x 2048 x 2000 55.6 against
        // 54.6).  Of the 32-deep ones the 128 x 256 tile is the faster (1536^3 53.4
        // against 52.6, 1024^3 equal).
        const long long slices64 =
            static_cast<long long>((M + 255) / 256) * ((N + 127) / 128) * ((K + 63) / 64);
        const long long tiles_w = static_cast<long long>((M + 127) / 128) * ((N + 255) / 256);
        const long long per_cta64 = tiles_w * ((K + 63) / 64) / sms;
        // The 256 x 128 entry spreads its refills except on tiles crossing M or N;
        // with such tiles and under 1.5 waves its all-burst twin is faster.
        const long long tiles_h = static_cast<long long>((M + 255) / 256) * ((N + 127) / 128);
        const bool ragged_h = (M % 256 != 0 || N % 128 != 0) && 2 * tiles_h < 3LL * sms;
        if (per_cta64 >= 44 && !ragged_h)
            name = "128x256x64_t8x16_s2_f2_v4";
        else if (slices64 >= 16LL * sms)
            name = ragged_h ? "256x128x64_t8x16_s2_f2_v4_burst" : "256x128x64_t8x16_s2_f2_v4";
        else
            name = "128x256x32_t8x16_s4_f2_v4";
    }
    else
        name = "128x256x32_t8x16_s3_f2_v1";
    return find_entry(name);
}

int choose_entry(const DeviceInfo& d, int M, int N, int K, const float* A, int lda,
                 const float* B, int ldb) {
    if (const char* force = std::getenv("SGEMM_FORCE_KERNEL")) {
        const int id = find_entry(force);
        if (id >= 0 && entry_fits(table()[id], A, lda, B, ldb) && d.occ[id] > 0)
            return id;
    }
    return choose_by_rules(d.sms, M, N, K, vec4_ok(A, lda, B, ldb));
}

// Time to store one BM x BN tile, in BK-deep slices of the same tile.  A slice
// is BM*BN*BK FMAs at about 100 per clock per SM; a store moves BM*BN*4 bytes at
// about 32 bytes per clock per SM (both measured on the 128 x 256 kernels, and
// both shared alike when several CTAs sit on one SM), so the ratio is ~12 / BK.
double store_cost_slices(const KernelEntry& e) { return 12.0 / e.bk; }

// schedule: 0 automatic, 1 data-parallel only, 2 stream-K whenever possible,
// 3 cluster split whenever possible.
// SGEMM_SK_GAP=<n> asks for that stream-K gap where it is allowed;
// SGEMM_GROUP_M=<n> sets the raster group height; SGEMM_CLUSTER=<S> asks for
// clusters of up to S CTAs per tile where allowed, 0 for none (tuning).
// `clusters` (null on the host-only checks): the entry's co-resident clusters of
// 2, 4 and 8 CTAs.  Where the automatic split means one wave of T clusters (T*S
// CTAs within the resident slots), it takes only a cluster size whose T clusters
// can all be resident at once: a second wave of clusters doubles the time
// (768 x 768 x 8192 on 128 x 256 x 32 tiles: 18 clusters of 8 where 15 fit ran
// below 38.3 TFLOP/s; stream-K over all 152 SMs instead, 56.0).  Splits that fill the SMs several times over
// by design are left alone.
void make_schedule(int sms, int occ, int entry, int schedule, Plan& p,
                   const std::array<int, 3>* clusters = nullptr) {
    const KernelEntry& e = table()[entry];
    int forced_gap = -1, group_m = 0, forced_cluster = -1;
    if (const char* g = std::getenv("SGEMM_SK_GAP")) forced_gap = std::atoi(g);
    if (const char* g = std::getenv("SGEMM_GROUP_M")) group_m = std::max(0, std::atoi(g));
    if (const char* g = std::getenv("SGEMM_CLUSTER")) forced_cluster = std::max(0, std::atoi(g));
    // The cp.async kernels sum cluster-split tiles in distributed shared memory;
    // the TMA-fed ones only take the stream-K reduction.
    int cluster_max = e.tma ? 0 : kMaxCluster;
    if (clusters != nullptr && schedule == 0 && forced_cluster < 0) {
        const long long T = static_cast<long long>((p.args.M + e.bm - 1) / e.bm) *
                            ((p.args.N + e.bn - 1) / e.bn);
        int l = 2;   // cluster_max = 2 << l
        while (cluster_max >= 2 && T * cluster_max <= static_cast<long long>(sms) * occ &&
               (*clusters)[l] < T) {
            cluster_max /= 2;
            --l;
        }
        if (cluster_max < 2) cluster_max = 0;
    }
    const SchedSizes z = plan_schedule(p.args, e.bm, e.bn, e.bk, sms, occ, schedule,
                                       store_cost_slices(e), forced_gap < 0 ? -1 : forced_gap,
                                       group_m, cluster_max, forced_cluster);
    p.ctas_per_sm = occ;
    p.split = z.split;
    p.ws_partial_bytes = z.partial_bytes;
}

int plan(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
         int ldc, int forced_entry, int schedule, Plan& p, const DeviceInfo** dinfo) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice", e);
        return SGEMM_ERR_UNSUPPORTED;
    }
    const DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != SGEMM_OK) return rc;
    *dinfo = d;
    const auto& t = table();
    int entry = forced_entry;
    if (entry >= 0) {
        if (entry >= static_cast<int>(t.size()) || !entry_fits(t[entry], A, lda, B, ldb) ||
            d->occ[entry] <= 0) {
            std::snprintf(t_last_error, sizeof(t_last_error),
                          "kernel %d cannot serve these operands", entry);
            return SGEMM_ERR_UNSUPPORTED;
        }
    } else {
        entry = choose_entry(*d, M, N, K, A, lda, B, ldb);
        if (entry < 0) {
            std::snprintf(t_last_error, sizeof(t_last_error), "no tile-table entry");
            return SGEMM_ERR_UNSUPPORTED;
        }
    }
    p.entry = entry;
    GemmArgs& a = p.args;
    a.M = M; a.N = N; a.K = K;
    a.A = A; a.B = B; a.C = C;
    a.lda = lda; a.ldb = ldb; a.ldc = ldc;
    a.c_vec = (aligned16(C) && ldc % 4 == 0) ? 1 : 0;
    make_schedule(d->sms, d->occ[entry], entry, schedule, p, &d->clusters[entry]);
    return SGEMM_OK;
}

// ----------------------------------------------------------------------------
// Workspaces owned by the library: one per (device, stream), grown on demand
// with the stream-ordered allocator so a resize never races in-flight work.
// A call holds its workspace's lock from the lookup until its launches are
// enqueued, so another host thread on the same stream cannot free the buffer
// (by growing it) between this call's lookup and its launch; calls on other
// streams take other locks.
// ----------------------------------------------------------------------------
struct Workspace {
    std::mutex mu;
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;   // guards the map itself; entries are stable until shutdown
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

int library_workspace(cudaStream_t stream, size_t need, void** out,
                      std::unique_lock<std::mutex>* hold) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice", e);
        return SGEMM_ERR_LAUNCH;
    }
    Workspace* wp = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_ws_mu);
        wp = &g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
    }
    std::unique_lock<std::mutex> wl(wp->mu);
    Workspace& w = *wp;
    if (w.bytes >= need) {
        *out = w.ptr;
        *hold = std::move(wl);
        return SGEMM_OK;
    }
    if (w.ptr) {
        e = cudaFreeAsync(w.ptr, stream);
        w.ptr = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess) {
            set_error("cudaFreeAsync", e);
            return SGEMM_ERR_WORKSPACE;
        }
    }
    const size_t bytes = std::max(need, static_cast<size_t>(1) << 20);
    e = cudaMallocAsync(&w.ptr, bytes, stream);
    if (e != cudaSuccess) {
        w.ptr = nullptr;
        set_error("cudaMallocAsync", e);
        return SGEMM_ERR_WORKSPACE;
    }
    w.bytes = bytes;
    *out = w.ptr;
    *hold = std::move(wl);
    return SGEMM_OK;
}

// C = beta * C over the M x N region (beta == 0 writes zeros without reading C):
// the whole product when K == 0 (the empty sum) or alpha == 0.
__global__ void scale_c_kernel(float* C, int M, int N, long long ldc, float beta) {
    const long long total = static_cast<long long>(M) * N;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long i = e / N, j = e - i * N;
        float* c = C + i * ldc + j;
        *c = beta == 0.0f ? 0.0f : beta * *c;
    }
}

int launch_scale(float* C, int M, int N, int ldc, float beta, cudaStream_t stream,
                 const DeviceInfo* d) {
    if (beta == 1.0f) return SGEMM_OK;
    const long long total = static_cast<long long>(M) * N;
    const int threads = 256;
    const long long blocks =
        std::min<long long>((total + threads - 1) / threads, static_cast<long long>(d->sms) * 8);
    scale_c_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(C, M, N, ldc, beta);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("scale_c_kernel launch", e);
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

int launch(const Plan& p, cudaStream_t stream) {
    const KernelEntry& e = table()[p.entry];
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.args.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(e.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(e.smem_bytes);
    cfg.stream = stream;
    // Programmatic dependent launch: the kernel may start while the stream's
    // previous kernel drains, and waits (griddepcontrol.wait) before touching
    // global memory.  SGEMM_PDL=0 launches it plainly (tuning).
    static const bool pdl = [] {
        const char* v = std::getenv("SGEMM_PDL");
        return v == nullptr || std::atoi(v) != 0;
    }();
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    if (p.args.cl_split > 1) {
        // Cluster split: CTAs t*S .. t*S+S-1 (one tile) form one cluster.
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(p.args.cl_split);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    GemmArgs args = p.args;
    void* params[] = {&args};
    FfmaTmaParams tp;
    void* tma_params[] = {&tp};
    if (e.tma) {
        // A: 32 (k) x BM boxes, 128-byte swizzle; B: BN (n) x BK boxes, no swizzle.
        tp.g = p.args;
        if (!encode_fp32_2d(&tp.ta, p.args.A, p.args.M, p.args.K, p.args.lda, 32, e.bm, 128) ||
            !encode_fp32_2d(&tp.tb, p.args.B, p.args.K, p.args.N, p.args.ldb, e.bn, e.bk, 0)) {
            std::snprintf(t_last_error, sizeof(t_last_error),
                          "%s: cuTensorMapEncodeTiled failed", e.name);
            return SGEMM_ERR_LAUNCH;
        }
    }
    cudaError_t err = cudaLaunchKernelExC(&cfg, e.kernel, e.tma ? tma_params : params);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) {
        set_error(e.name, err);
        return SGEMM_ERR_LAUNCH;
    }
    if (p.args.sk_tiles > 0 && p.args.cl_split <= 1) {
        err = launch_sk_reduce(p.args, e.bm, e.bn, p.sms, stream);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (err != cudaSuccess) {
            set_error("sk_reduce_kernel", err);
            return SGEMM_ERR_LAUNCH;
        }
    }
    return SGEMM_OK;
}

// Row-by-row copy of a rows x cols matrix into a buffer whose leading dimension
// ldd is a multiple of 4 (16-byte rows), for operands whose own rows are not
// 16-byte aligned.  Each thread moves 4 consecutive elements of one row.
__global__ void pack_rows_kernel(const float* __restrict__ src, long long lds, int rows,
                                 int cols, float* __restrict__ dst, long long ldd) {
    const int c = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (c >= cols) return;
    for (int r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* s = src + r * lds + c;
        float4 v;
        v.x = __ldg(s);
        v.y = c + 1 < cols ? __ldg(s + 1) : 0.0f;
        v.z = c + 2 < cols ? __ldg(s + 2) : 0.0f;
        v.w = c + 3 < cols ? __ldg(s + 3) : 0.0f;
        *reinterpret_cast<float4*>(dst + r * ldd + c) = v;
    }
}

int launch_pack(const float* src, long long lds, int rows, int cols, float* dst, long long ldd,
                cudaStream_t stream) {
    const dim3 grid((cols / 4 + 1 + 255) / 256, std::min(rows, 65535));
    pack_rows_kernel<<<grid, 256, 0, stream>>>(src, lds, rows, cols, dst, ldd);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("pack_rows_kernel launch", e);
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

// Y = X^T: X is rows x cols (leading dimension ldx), Y is cols x rows (leading
// dimension ldy, a multiple of 4, with Y 16-byte aligned; its padding columns are
// not written).  64 x 64 tiles through shared memory (row stride 65), 256
// threads: each moves four 16-byte chunks in and four out per tile, so a CTA has
// 16 KB of loads in flight.  X is read as float4 when its rows are 16-byte
// aligned, else element by element.  HBM-bound.
__global__ void __launch_bounds__(256) transpose_kernel(const float* __restrict__ X,
                                                        long long ldx, int rows, int cols,
                                                        float* __restrict__ Y, long long ldy,
                                                        int x_vec) {
    constexpr int T = 64;
    __shared__ float t[T][T + 1];
    const long long tiles_c = (cols + T - 1) / T;
    const long long tiles = tiles_c * ((rows + T - 1) / T);
    for (long long tt = blockIdx.x; tt < tiles; tt += gridDim.x) {
        const int r0 = static_cast<int>(tt / tiles_c) * T;
        const int c0 = static_cast<int>(tt % tiles_c) * T;
#pragma unroll
        for (int e = threadIdx.x; e < T * T / 4; e += 256) {
            const int r = e / (T / 4), c4 = (e % (T / 4)) * 4;
            const int gr = r0 + r, gc = c0 + c4;
            if (gr >= rows) continue;
            const float* src = X + gr * ldx + gc;
            if (x_vec && gc + 3 < cols) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                t[r][c4] = v.x; t[r][c4 + 1] = v.y; t[r][c4 + 2] = v.z; t[r][c4 + 3] = v.w;
            } else {
                for (int q = 0; q < 4 && gc + q < cols; ++q) t[r][c4 + q] = src[q];
            }
        }
        __syncthreads();
#pragma unroll
        for (int e = threadIdx.x; e < T * T / 4; e += 256) {
            const int c = e / (T / 4), r4 = (e % (T / 4)) * 4;
            const int gy = c0 + c, gx = r0 + r4;   // Y[gy][gx..gx+3] = X[gx..gx+3][gy]
            if (gy >= cols) continue;
            float* dst = Y + gy * ldy + gx;
            if (gx + 3 < rows) {
                *reinterpret_cast<float4*>(dst) =
                    make_float4(t[r4][c], t[r4 + 1][c], t[r4 + 2][c], t[r4 + 3][c]);
            } else {
                for (int q = 0; q < 4 && gx + q < rows; ++q) dst[q] = t[r4 + q][c];
            }
        }
        __syncthreads();
    }
}

int launch_transpose(const float* X, long long ldx, int rows, int cols, float* Y, long long ldy,
                     int sms, cudaStream_t stream) {
    const long long tiles = ((rows + 63) / 64) * static_cast<long long>((cols + 63) / 64);
    const int grid = static_cast<int>(std::max(1LL, std::min<long long>(tiles, 8LL * sms)));
    const int x_vec = aligned16(X) && ldx % 4 == 0;
    transpose_kernel<<<grid, 256, 0, stream>>>(X, ldx, rows, cols, Y, ldy, x_vec);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("transpose_kernel launch", e);
        return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
}

// Problems whose A or B rows are not 16-byte aligned are worth copying to aligned
// buffers first once K is not short: the 4-byte-load kernels then run 15-40 %
// slower than the 16-byte ones (copy included, 1024^3 29.7 against 36.4 TFLOP/s,
// 1536 x 1536 x 768 34.5 against 43.9, 768 x 768 x 3000 27.7 against 41.3), while
// with K of a few hundred they run as fast and the copy is pure cost (2048 x 2048 x
// 511: 33.9 against 32.5).  The copy moves 8 bytes per operand element and takes
// two launches, so the product must be large enough to pay for them.
constexpr double kPackMinMacs = 5.0e8;   // M * N * K
constexpr int kPackMinK = 768;

// Operand staging in the library workspace: a transposed operand is always
// transposed into a row-major buffer; a misaligned one of a large problem is
// copied row by row.  Staged buffers have 16-byte-aligned rows.
struct PackPlan {
    bool pack_a = false, pack_b = false;
    bool trans_a = false, trans_b = false;
    int lda = 0, ldb = 0;         // leading dimensions the kernels will see
    size_t bytes_a = 0, bytes_b = 0;
    const float* plan_a = nullptr;
    const float* plan_b = nullptr;
};

PackPlan pack_plan(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                   bool library_ws, int forced_entry, int transa, int transb) {
    PackPlan q;
    q.trans_a = transa != 0;
    q.trans_b = transb != 0;
    // Each non-transposed operand is packed on its own: a transposed partner is
    // staged aligned anyway, so the other one alone decides the load width.
    const bool pack = library_ws && forced_entry < 0 && K >= kPackMinK &&
                      static_cast<double>(M) * N * K >= kPackMinMacs;
    q.pack_a = q.trans_a || (pack && !(aligned16(A) && lda % 4 == 0));
    q.pack_b = q.trans_b || (pack && !(aligned16(B) && ldb % 4 == 0));
    q.lda = q.pack_a ? (K + 3) / 4 * 4 : lda;
    q.ldb = q.pack_b ? (N + 3) / 4 * 4 : ldb;
    q.bytes_a = q.pack_a ? align_up(static_cast<size_t>(M) * q.lda * 4, kWsAlign) : 0;
    q.bytes_b = q.pack_b ? align_up(static_cast<size_t>(K) * q.ldb * 4, kWsAlign) : 0;
    // Alignment-only stand-ins for the staged buffers while planning.
    q.plan_a = q.pack_a ? reinterpret_cast<const float*>(uintptr_t{256}) : A;
    q.plan_b = q.pack_b ? reinterpret_cast<const float*>(uintptr_t{256} << 20) : B;
    return q;
}

// Common body of the run entry points: C = alpha * op(A).op(B) + beta * C (the
// plain entry points pass alpha = 1, beta = 0).  library_ws selects the
// library-owned workspace; otherwise the caller's (ws, ws_bytes) serves the
// split tiles and nothing is staged.
int run_impl(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
             float beta, float* C, int ldc, int forced_entry, int schedule, void* ws,
             size_t ws_bytes, bool library_ws, cudaStream_t stream, int transa = 0,
             int transb = 0) {
    int rc = check_args_op(transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0) return SGEMM_OK;
    Plan p;
    const DeviceInfo* d = nullptr;
    if (K == 0 || alpha == 0.0f) {
        // The product term vanishes (empty sum, or alpha = 0): A and B are not read.
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            set_error("cudaGetDevice", e);
            return SGEMM_ERR_UNSUPPORTED;
        }
        rc = device_info(dev, &d);
        if (rc != SGEMM_OK) return rc;
        return launch_scale(C, M, N, ldc, beta, stream, d);
    }
    // Staging (library workspace only): transposed operands, and misaligned ones
    // of large problems, are copied to aligned row-major buffers at the front of
    // the workspace and the plan is made for them.
    if ((transa || transb) && !library_ws) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "transposed operands need the library workspace");
        return SGEMM_ERR_UNSUPPORTED;
    }
    const PackPlan q = pack_plan(M, N, K, A, lda, B, ldb, library_ws, forced_entry, transa,
                                 transb);
    const bool pack = q.pack_a || q.pack_b;
    const bool pack_a = q.pack_a, pack_b = q.pack_b;
    const int lda_p = q.lda, ldb_p = q.ldb;
    const size_t bytes_a = q.bytes_a, bytes_b = q.bytes_b;
    rc = plan(M, N, K, q.plan_a, lda_p, q.plan_b, ldb_p, C, ldc, forced_entry, schedule, p, &d);
    if (rc != SGEMM_OK) return rc;
    p.args.A = A;
    p.args.B = B;
    p.args.alpha = alpha;
    p.args.beta = beta;
    p.args.status = status_word_ptr();
    p.args.epi = (beta != 0.0f) ? kEpiAlphaBeta : (alpha != 1.0f ? kEpiAlpha : kEpiPlain);
    std::unique_lock<std::mutex> ws_hold;   // the library workspace, until launched
    if (pack) {
        void* base = nullptr;
        rc = library_workspace(stream, bytes_a + bytes_b + p.ws_partial_bytes, &base,
                               &ws_hold);
        if (rc != SGEMM_OK) return rc;
        char* w = static_cast<char*>(base);
        if (pack_a) {
            float* pa = reinterpret_cast<float*>(w);
            rc = q.trans_a ? launch_transpose(A, lda, K, M, pa, lda_p, d->sms, stream)
                           : launch_pack(A, lda, M, K, pa, lda_p, stream);
            if (rc != SGEMM_OK) return rc;
            p.args.A = pa;
        }
        if (pack_b) {
            float* pb = reinterpret_cast<float*>(w + bytes_a);
            rc = q.trans_b ? launch_transpose(B, ldb, N, K, pb, ldb_p, d->sms, stream)
                           : launch_pack(B, ldb, K, N, pb, ldb_p, stream);
            if (rc != SGEMM_OK) return rc;
            p.args.B = pb;
        }
        p.args.ws_partial = reinterpret_cast<float*>(w + bytes_a + bytes_b);
        p.sms = d->sms;
        return launch(p, stream);
    }
    const size_t need = p.ws_partial_bytes;
    if (need > 0) {
        void* base = nullptr;
        if (library_ws) {
            rc = library_workspace(stream, need, &base, &ws_hold);
            if (rc != SGEMM_OK) return rc;
        } else {
            if (ws == nullptr || ws_bytes < need || !aligned16(ws)) {
                std::snprintf(t_last_error, sizeof(t_last_error),
                              "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
                return SGEMM_ERR_WORKSPACE;
            }
            base = ws;
        }
        p.args.ws_partial = static_cast<float*>(base);
    }
    p.sms = d->sms;
    return launch(p, stream);
}

void fill_config(const Plan& p, sgemm_config* out) {
    const KernelEntry& e = table()[p.entry];
    out->bm = e.bm; out->bn = e.bn; out->bk = e.bk;
    out->wm = e.wm; out->wn = e.wn; out->tm = e.tm; out->tn = e.tn;
    out->stages = e.stages; out->threads = e.threads; out->smem_bytes = e.smem_bytes;
    out->split_k = p.split;
    out->kernel_id = p.entry;
    out->vec = e.vec;
    out->grid = p.args.grid;
    out->tiles = p.args.tiles_m * p.args.tiles_n;
    out->sk_tiles = p.args.sk_tiles;
    out->ctas_per_sm = p.ctas_per_sm;
    out->fma2 = e.fma2;
    out->sk_gap = p.args.sk_gap;
    out->cluster = p.args.cl_split > 1 ? p.args.cl_split : 0;
}

// Walks every CTA's flat slice list exactly as the kernel does and checks the
// schedule: each (tile, k-slice) is computed once, tile origins are distinct and
// inside C, every split tile's contributors write slots 0/1 only and number
// exactly what the kernel's owner formula expects.
int check_schedule(const Plan& p, char* why, size_t why_len) {
    const KernelEntry& e = table()[p.entry];
    const GemmArgs& a = p.args;
    const long long T = static_cast<long long>(a.tiles_m) * a.tiles_n;
    const int KT = a.KT, G = a.grid;
    auto fail = [&](const char* msg, long long x, long long y) {
        std::snprintf(why, why_len, "%s (%lld, %lld)", msg, x, y);
        return SGEMM_ERR_INVALID_ARG;
    };
    if (G <= 0 || a.dp_tiles + a.sk_tiles != T) return fail("tile count", G, T);
    const int S = a.cl_split;
    if (S > 1) {
        // Cluster split: T clusters of S CTAs, CTA t*S+r holds a non-empty piece
        // of tile t only, pieces in rank order, the cluster size divides BM.
        if (S > kMaxCluster || (S & (S - 1)) != 0) return fail("cluster size", S, 0);
        if (a.dp_tiles != 0 || static_cast<long long>(a.sk_tiles) * S != G || a.sk_gap != 0)
            return fail("cluster grid", G, a.sk_tiles);
        if (e.bm % S != 0 || e.tma) return fail("cluster sum unsupported", e.bm, S);
        for (int g = 0; g < G; ++g) {
            const CtaWork w = make_work(a, g);
            if (w.total <= 0) return fail("CTA without work", g, w.total);
            // The kernels' division-free form of the same work.
            const CtaWork wc = make_cluster_work(a, g);
            if (wc.u0 != w.u0 || wc.u1 != w.u1 || wc.total != w.total || wc.dp_iters != 0 ||
                w.dp_iters != 0)
                return fail("cluster work differs from the stream-K formula", g, wc.u0);
            Cursor c;
            c.seek(w, 0);
            const int want_tile = g / S;
            if (c.tile != want_tile || c.kt_begin != static_cast<int>(
                                           static_cast<long long>(KT) * (g % S) / S) ||
                c.kt_end != static_cast<int>(static_cast<long long>(KT) * (g % S + 1) / S) ||
                w.total != c.kt_end - c.kt_begin)
                return fail("cluster piece", g, c.tile);
        }
    }
    if (a.sk_tiles > 0 && a.sk_iters < G) return fail("stream-K range empty", a.sk_iters, G);
    if (a.sk_tiles > G) return fail("more split tiles than CTAs", a.sk_tiles, G);
    std::vector<unsigned char> cover(static_cast<size_t>(T) * KT, 0);
    std::vector<int> contrib(static_cast<size_t>(a.sk_tiles), 0);
    for (int g = 0; g < G; ++g) {
        const CtaWork w = make_work(a, g);
        if (w.total <= 0) return fail("CTA without work", g, w.total);
        Cursor c;
        c.seek(w, 0);
        for (long long it = 0; it < w.total; ++it) {
            if (c.tile < 0 || c.tile >= T || c.kt < 0 || c.kt >= KT || c.kt < c.kt_begin ||
                c.kt >= c.kt_end)
                return fail("cursor out of range", c.tile, c.kt);
            if (++cover[static_cast<size_t>(c.tile) * KT + c.kt] != 1)
                return fail("slice computed twice", c.tile, c.kt);
            if (c.kt + 1 == c.kt_end && !(c.kt_begin == 0 && c.kt_end == KT)) {
                const int t = c.tile - a.dp_tiles;
                if (t < 0 || t >= a.sk_tiles) return fail("partial outside split tiles", g, t);
                const int slot = sk_slot(w, t);
                if (slot < 0 || slot > 1) return fail("slot out of range", g, slot);
                ++contrib[static_cast<size_t>(t)];
            }
            c.advance(w);
        }
    }
    for (size_t i = 0; i < cover.size(); ++i)
        if (cover[i] != 1) return fail("slice never computed", static_cast<long long>(i / KT),
                                       static_cast<long long>(i % KT));
    for (int t = 0; t < a.sk_tiles; ++t) {
        const long long tb = static_cast<long long>(t) * KT;
        const int g0 = sk_owner(a, tb), g1 = sk_owner(a, tb + KT - 1);
        if (contrib[t] == 0) {
            if (g0 != g1) return fail("whole split tile with several owners", t, g1 - g0);
            continue;
        }
        if (contrib[t] != g1 - g0 + 1) return fail("contributor count", t, contrib[t]);
        if (contrib[t] > kMaxSplit) return fail("too many contributors", t, contrib[t]);
        for (int gg = g0; gg <= g1; ++gg) {
            const int sl = t - static_cast<int>(sk_begin(a, gg) / KT);
            if (sl < 0 || sl > 1) return fail("reduction slot out of range", t, gg);
        }
    }
    std::vector<unsigned char> seen(static_cast<size_t>(T), 0);
    for (long long tile = 0; tile < T; ++tile) {
        int m0 = 0, n0 = 0;
        tile_origin(a, static_cast<int>(tile), e.bm, e.bn, m0, n0);
        if (m0 < 0 || n0 < 0 || m0 >= a.M || n0 >= a.N || m0 % e.bm || n0 % e.bn)
            return fail("tile origin outside C", m0, n0);
        const size_t id = static_cast<size_t>(m0 / e.bm) * a.tiles_n + n0 / e.bn;
        if (seen[id]++) return fail("tile origin repeated", m0, n0);
    }
    return SGEMM_OK;
}

}  // namespace

void set_cuda_error(const char* what, cudaError_t e) { set_error(what, e); }

int check_sizes(int M, int N, int K) { return check_dims(M, N, K); }

int check_operands(int transa, int transb, int M, int N, int K, const float* A, int lda,
                   const float* B, int ldb, const float* C, int ldc) {
    return check_args_op(transa, transb, M, N, K, A, lda, B, ldb, C, ldc);
}

void set_last_error_message(const char* msg) {
    std::snprintf(t_last_error, sizeof(t_last_error), "%s", msg);
}

}  // namespace sgemm

using namespace sgemm;

extern "C" {

int sgemm_run(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
              int ldc, sgemm_stream_t stream) {
    return run_impl(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, -1, 0, nullptr, 0, true,
                    reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_run_ex(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                 int ldb, float beta, float* C, int ldc, int kernel_id, int schedule,
                 sgemm_stream_t stream) {
    if (kernel_id < -1 || schedule < 0 || schedule > 3) {
        std::snprintf(t_last_error, sizeof(t_last_error), "bad kernel_id %d or schedule %d",
                      kernel_id, schedule);
        return kernel_id < -1 ? SGEMM_ERR_UNSUPPORTED : SGEMM_ERR_INVALID_ARG;
    }
    if (!(alpha == alpha) || !(beta == beta)) {
        std::snprintf(t_last_error, sizeof(t_last_error), "alpha or beta is NaN");
        return SGEMM_ERR_INVALID_ARG;
    }
    return run_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, kernel_id, schedule, nullptr,
                    0, true, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_run_op(int transa, int transb, int M, int N, int K, float alpha, const float* A,
                 int lda, const float* B, int ldb, float beta, float* C, int ldc,
                 sgemm_stream_t stream) {
    if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1)) {
        std::snprintf(t_last_error, sizeof(t_last_error), "transa=%d transb=%d (0 or 1)", transa,
                      transb);
        return SGEMM_ERR_INVALID_ARG;
    }
    if (!(alpha == alpha) || !(beta == beta)) {
        std::snprintf(t_last_error, sizeof(t_last_error), "alpha or beta is NaN");
        return SGEMM_ERR_INVALID_ARG;
    }
    return run_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, -1, 0, nullptr, 0, true,
                    reinterpret_cast<cudaStream_t>(stream), transa, transb);
}

int sgemm_run_ws(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                 float* C, int ldc, void* ws, size_t ws_bytes, sgemm_stream_t stream) {
    return run_impl(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, -1, 0, ws, ws_bytes, false,
                    reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_run_with(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                   float* C, int ldc, int kernel_id, int schedule, sgemm_stream_t stream) {
    if (kernel_id < -1 || schedule < 0 || schedule > 3) {
        std::snprintf(t_last_error, sizeof(t_last_error), "bad kernel_id %d or schedule %d",
                      kernel_id, schedule);
        return kernel_id < -1 ? SGEMM_ERR_UNSUPPORTED : SGEMM_ERR_INVALID_ARG;
    }
    return run_impl(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, kernel_id, schedule, nullptr, 0,
                    true,
                    reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_workspace_size(int M, int N, int K, int lda, int ldb, int ldc, const float* A,
                         const float* B, const float* C, size_t* out_bytes) {
    if (out_bytes == nullptr) return SGEMM_ERR_INVALID_ARG;
    *out_bytes = 0;
    // Alignment-only use of the pointers: substitute aligned stand-ins for NULL.
    const float* pa = A ? A : reinterpret_cast<const float*>(uintptr_t{256});
    const float* pb = B ? B : reinterpret_cast<const float*>(uintptr_t{256} << 20);
    const float* pc = C ? C : reinterpret_cast<const float*>(uintptr_t{256} << 40);
    if (M < 0 || N < 0 || K < 0 || lda < std::max(K, 1) || ldb < std::max(N, 1) ||
        ldc < std::max(N, 1))
        return SGEMM_ERR_INVALID_ARG;
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0 || K == 0) return SGEMM_OK;
    Plan p;
    const DeviceInfo* d = nullptr;
    const int rc = plan(M, N, K, pa, lda, pb, ldb, const_cast<float*>(pc), ldc, -1, 0, p, &d);
    if (rc != SGEMM_OK) return rc;
    *out_bytes = p.ws_partial_bytes;
    return SGEMM_OK;
}

int sgemm_query_config(int M, int N, int K, int lda, int ldb, int ldc, const float* A,
                       const float* B, const float* C, sgemm_config* out) {
    if (out == nullptr) return SGEMM_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    const float* pa = A ? A : reinterpret_cast<const float*>(uintptr_t{256});
    const float* pb = B ? B : reinterpret_cast<const float*>(uintptr_t{256} << 20);
    const float* pc = C ? C : reinterpret_cast<const float*>(uintptr_t{256} << 40);
    if (M <= 0 || N <= 0 || K <= 0 || lda < K || ldb < N || ldc < N)
        return SGEMM_ERR_INVALID_ARG;
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    Plan p;
    const DeviceInfo* d = nullptr;
    const PackPlan q = pack_plan(M, N, K, pa, lda, pb, ldb, true, -1, 0, 0);
    const int rc =
        plan(M, N, K, q.plan_a, q.lda, q.plan_b, q.ldb, const_cast<float*>(pc), ldc, -1, 0, p, &d);
    if (rc != SGEMM_OK) return rc;
    fill_config(p, out);
    out->packed = (q.pack_a ? 1 : 0) | (q.pack_b ? 2 : 0);
    return SGEMM_OK;
}

int sgemm_schedule_check(int M, int N, int K, int kernel_id, int sms, int ctas_per_sm,
                         int schedule, sgemm_config* out) {
    if (M <= 0 || N <= 0 || K <= 0 || sms <= 0 || ctas_per_sm <= 0 || schedule < 0 ||
        schedule > 3 || kernel_id < 0 || kernel_id >= static_cast<int>(table().size()))
        return SGEMM_ERR_INVALID_ARG;
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    Plan p;
    p.entry = kernel_id;
    p.args.M = M; p.args.N = N; p.args.K = K;
    make_schedule(sms, ctas_per_sm, kernel_id, schedule, p);
    if (out) fill_config(p, out);
    return check_schedule(p, t_last_error, sizeof(t_last_error));
}

int sgemm_choose_check(int M, int N, int K, int lda, int ldb, int a_offset, int b_offset,
                       int sms, int* kernel_id, int* packed) {
    if (M <= 0 || N <= 0 || K <= 0 || lda < K || ldb < N || sms <= 0 || a_offset < 0 ||
        a_offset > 3 || b_offset < 0 || b_offset > 3 || kernel_id == nullptr)
        return SGEMM_ERR_INVALID_ARG;
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    // Stand-ins that carry only the operands' alignment.
    const float* pa = reinterpret_cast<const float*>(uintptr_t{256} + 4u * a_offset);
    const float* pb = reinterpret_cast<const float*>((uintptr_t{256} << 20) + 4u * b_offset);
    const PackPlan q = pack_plan(M, N, K, pa, lda, pb, ldb, true, -1, 0, 0);
    *kernel_id = choose_by_rules(sms, M, N, K, vec4_ok(q.plan_a, q.lda, q.plan_b, q.ldb));
    if (packed) *packed = (q.pack_a ? 1 : 0) | (q.pack_b ? 2 : 0);
    return *kernel_id >= 0 ? SGEMM_OK : SGEMM_ERR_UNSUPPORTED;
}

int sgemm_tf32x3_workspace_size(int M, int N, int K, size_t* out_bytes) {
    if (out_bytes == nullptr || M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    *out_bytes = tf32x3_workspace_bytes(M, N, K);
    return SGEMM_OK;
}

int sgemm_tf32x3_run_ex(int M, int N, int K, float alpha, const float* A, int lda,
                        const float* B, int ldb, float beta, float* C, int ldc, void* ws,
                        size_t ws_bytes, sgemm_stream_t stream) {
    int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (rc != SGEMM_OK) return rc;
    if (!(alpha == alpha) || !(beta == beta)) {
        std::snprintf(t_last_error, sizeof(t_last_error), "alpha or beta is NaN");
        return SGEMM_ERR_INVALID_ARG;
    }
    if (M == 0 || N == 0) return SGEMM_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_error("cudaGetDevice", e);
        return SGEMM_ERR_UNSUPPORTED;
    }
    const DeviceInfo* d = nullptr;
    rc = device_info(dev, &d);
    if (rc != SGEMM_OK) return rc;
    if (K == 0 || alpha == 0.0f) return launch_scale(C, M, N, ldc, beta, s, d);
    const size_t need = tf32x3_workspace_bytes(M, N, K);
    std::unique_lock<std::mutex> ws_hold;   // the library workspace, until launched
    if (ws == nullptr) {
        rc = library_workspace(s, need, &ws, &ws_hold);
        if (rc != SGEMM_OK) return rc;
        ws_bytes = need;
    } else if (ws_bytes < need || !aligned16(ws)) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
        return SGEMM_ERR_WORKSPACE;
    }
    const int c_vec = (aligned16(C) && ldc % 4 == 0) ? 1 : 0;
    // A that TMA can read (16-byte aligned rows) serves as its own hi part, so the
    // split writes only Alo for it.  SGEMM_TF32X3_SPLIT_A=1 writes Ahi anyway.
    const char* split_env = std::getenv("SGEMM_TF32X3_SPLIT_A");
    const bool force_split = split_env != nullptr && std::atoi(split_env) != 0;
    const bool a_direct = !force_split && aligned16(A) && lda % 4 == 0;
    rc = tf32x3_prepare(M, N, K, A, lda, B, ldb, ws, ws_bytes, d->sms, s, !a_direct);
    g_launches.fetch_add(1, std::memory_order_relaxed);   // split_kernel
    if (rc != SGEMM_OK) return rc;
    int n = 0;
    rc = tf32x3_multiply(M, N, K, alpha, beta, C, ldc, c_vec, ws, ws_bytes, d->sms, s, &n,
                         a_direct ? A : nullptr, lda);
    g_launches.fetch_add(n, std::memory_order_relaxed);
    return rc;
}

int sgemm_tf32x3_prepare(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                         void* ws, size_t ws_bytes, sgemm_stream_t stream) {
    int rc = check_args(M, N, K, A, lda, B, ldb, reinterpret_cast<const float*>(ws), std::max(N, 1));
    if (rc != SGEMM_OK) return rc;
    if (M == 0 || N == 0 || K == 0) return SGEMM_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED;
    const DeviceInfo* d = nullptr;
    rc = device_info(dev, &d);
    if (rc != SGEMM_OK) return rc;
    if (!aligned16(ws)) return SGEMM_ERR_WORKSPACE;
    rc = tf32x3_prepare(M, N, K, A, lda, B, ldb, ws, ws_bytes,
                        d->sms, reinterpret_cast<cudaStream_t>(stream));
    g_launches.fetch_add(1, std::memory_order_relaxed);   // split_kernel
    return rc;
}

int sgemm_tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C, int ldc,
                          const void* ws, size_t ws_bytes, sgemm_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || ldc < std::max(N, 1) || (M > 0 && N > 0 && C == nullptr) ||
        !(alpha == alpha) || !(beta == beta)) {
        std::snprintf(t_last_error, sizeof(t_last_error), "invalid argument");
        return SGEMM_ERR_INVALID_ARG;
    }
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return SGEMM_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED;
    const DeviceInfo* d = nullptr;
    int rc = device_info(dev, &d);
    if (rc != SGEMM_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0 || alpha == 0.0f) return launch_scale(C, M, N, ldc, beta, s, d);
    if (ws == nullptr || !aligned16(ws)) return SGEMM_ERR_WORKSPACE;
    const int c_vec = (aligned16(C) && ldc % 4 == 0) ? 1 : 0;
    int n = 0;
    rc = tf32x3_multiply(M, N, K, alpha, beta, C, ldc, c_vec, const_cast<void*>(ws), ws_bytes,
                         d->sms, s, &n);
    g_launches.fetch_add(n, std::memory_order_relaxed);
    return rc;
}

int sgemm_tf32x3_query_config(int M, int N, int K, sgemm_config* out) {
    if (out == nullptr || M <= 0 || N <= 0 || K <= 0) return SGEMM_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    if (check_dims(M, N, K) != SGEMM_OK) return SGEMM_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED;
    const DeviceInfo* d = nullptr;
    const int rc = device_info(dev, &d);
    if (rc != SGEMM_OK) return rc;
    return tf32x3_query(M, N, K, d->sms, out);
}

int sgemm_tf32x3_run(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                     float* C, int ldc, sgemm_stream_t stream) {
    return sgemm_tf32x3_run_ex(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, nullptr, 0, stream);
}

int sgemm_device_status(void) {
    int flag = 0;
    const int rc = read_and_clear_status(&flag);
    if (rc != SGEMM_OK) {
        std::snprintf(t_last_error, sizeof(t_last_error), "cannot read the device status word");
        return rc;
    }
    if (flag) {
        std::snprintf(t_last_error, sizeof(t_last_error),
                      "a bounded wait in a TMA-fed kernel gave up");
        return SGEMM_ERR_TIMEOUT;
    }
    return SGEMM_OK;
}

int sgemm_selftest_bounded_wait(int limit_ms) {
    if (limit_ms < 1 || limit_ms > 10000) return SGEMM_ERR_INVALID_ARG;
    const int rc = run_wait_selftest(limit_ms);
    if (rc != SGEMM_OK) {
        std::snprintf(t_last_error, sizeof(t_last_error), "self-test kernel failed to run");
        return rc;
    }
    return sgemm_device_status();
}

int sgemm_num_kernels(void) { return static_cast<int>(table().size()); }

int sgemm_kernel_info(int kernel_id, sgemm_config* out) {
    if (out == nullptr) return SGEMM_ERR_INVALID_ARG;
    if (kernel_id < 0 || kernel_id >= static_cast<int>(table().size()))
        return SGEMM_ERR_UNSUPPORTED;
    std::memset(out, 0, sizeof(*out));
    const KernelEntry& e = table()[kernel_id];
    out->bm = e.bm; out->bn = e.bn; out->bk = e.bk;
    out->wm = e.wm; out->wn = e.wn; out->tm = e.tm; out->tn = e.tn;
    out->stages = e.stages; out->threads = e.threads; out->smem_bytes = e.smem_bytes;
    out->kernel_id = kernel_id;
    out->vec = e.vec;
    out->fma2 = e.fma2;
    return SGEMM_OK;
}

const char* sgemm_kernel_name(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= static_cast<int>(table().size())) return "";
    return table()[kernel_id].name;
}

const char* sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG";
        case SGEMM_ERR_ALIGNMENT: return "SGEMM_ERR_ALIGNMENT";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH";
        case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT";
        case SGEMM_ERR_WORKSPACE: return "SGEMM_ERR_WORKSPACE";
        default: return "SGEMM_ERR_UNKNOWN";
    }
}

const char* sgemm_last_error(void) { return t_last_error; }

uint64_t sgemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int sgemm_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int rc = SGEMM_OK;
    for (auto& kv : g_ws) {
        if (kv.second.ptr) {
            int prev = 0;
            cudaGetDevice(&prev);
            cudaSetDevice(kv.first.first);
            const cudaError_t e = cudaFree(kv.second.ptr);
            cudaSetDevice(prev);
            if (e != cudaSuccess) {
                set_error("cudaFree", e);
                rc = SGEMM_ERR_LAUNCH;
            }
        }
    }
    g_ws.clear();
    shutdown_host_pipes();
    forget_noalloc_scratch();
    forget_tf32x3_attributes();
    {
        // Kernel attributes live in the device's context: a context made after a
        // device reset needs them set again, so the per-device facts are redone.
        std::lock_guard<std::mutex> ld(g_dev_mu);
        g_dev.clear();
    }
    return rc;
}

}  // extern "C"
