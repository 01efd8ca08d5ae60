// Second phase of a stream-K launch: sums the partial tiles of every split tile.
//
// Each CTA of the main kernel that worked on part of a split tile's K range
// wrote its partial BM x BN sum to its own workspace slot.  Here every split
// tile is cut into `chunks` pieces and each piece is reduced by one CTA, so all
// SMs share the (L2-resident) partial data.  Partials are added in increasing
// CTA order, i.e. in increasing k, which fixes the summation order: the result
// does not depend on timing.  The schedule formulas are the ones the main
// kernel used (sgemm_sched.cuh).
#include <mutex>
#include <vector>

#include "sgemm_epilogue.cuh"
#include "sgemm_internal.h"
#include "sgemm_sched.cuh"

namespace sgemm {

namespace {

constexpr int kReduceThreads = 256;
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kReduceThreads) sk_reduce_kernel(const GemmArgs a, int bm,
                                                                   int bn, int chunks) {
    __shared__ const float4* s_src[kMaxSplit];
    // Launched as a programmatic dependent of the main kernel.  The contributor
    // list below depends on the launch arguments only, so it is worked out while
    // the main kernel finishes; griddepcontrol.wait comes before the first read
    // of anything that kernel wrote.
    const int t = blockIdx.x / chunks, part = blockIdx.x - t * chunks;
    const long long tb = static_cast<long long>(t) * a.KT;
    const int g0 = sk_owner(a, tb);
    const int g1 = sk_owner(a, tb + a.KT - 1);
    const int n = g1 - g0 + 1;  // contributors, in increasing k order
    if (n <= 1) {
        // One CTA held the whole K range and stored the tile itself.  Still wait
        // for the main kernel: a kernel launched as a programmatic dependent of
        // this one relies on the main kernel having completed when this grid has.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const long long tile_floats = static_cast<long long>(bm) * bn;
    for (int i = threadIdx.x; i < n; i += kReduceThreads) {
        const int gg = g0 + i;
        const int slot = t - static_cast<int>(sk_begin(a, gg) / a.KT);
        s_src[i] = reinterpret_cast<const float4*>(
            a.ws_partial + (static_cast<long long>(gg) * 2 + slot) * tile_floats);
    }
    __syncthreads();
    int m0, n0;
    tile_origin(a, a.dp_tiles + t, bm, bn, m0, n0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n4 = bm * bn / 4;  // float4 per tile
    const int per = (n4 + chunks - 1) / chunks;
    const int e_end = min(n4, (part + 1) * per);
    for (int e = part * per + threadIdx.x; e < e_end; e += kReduceThreads) {
        // Up to kBatch loads in flight per thread; the additions still follow
        // contributor order 0, 1, 2, ... exactly.
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = 0; i0 < n; i0 += kBatch) {
            float4 q[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < n) q[j] = __ldcg(s_src[i0 + j] + e);
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (i0 + j < n) {
                    s.x += q[j].x;
                    s.y += q[j].y;
                    s.z += q[j].z;
                    s.w += q[j].w;
                }
        }
        const int r = (4 * e) / bn, c = (4 * e) - r * bn;
        const int gm = m0 + r, gn = n0 + c;
        if (gm >= a.M) continue;
        store_c4(a, a.C + gm * a.ldc, gn, s);
    }
}

}  // namespace

int reduce_chunks(int bm, int bn, int sk_tiles, int sms) {
    const int n4 = bm * bn / 4;
    int chunks = (4 * sms + sk_tiles - 1) / sk_tiles;          // about four CTAs per SM
    const int max_chunks = (n4 + kReduceThreads - 1) / kReduceThreads;
    if (chunks > max_chunks) chunks = max_chunks;
    return chunks < 1 ? 1 : chunks;
}

cudaError_t launch_sk_reduce(const GemmArgs& a, int bm, int bn, int sms, cudaStream_t stream) {
    // Same shared-memory carveout preference as the GEMM kernels, so the SMs need
    // not be reconfigured between the two launches.  It is an attribute of the
    // kernel in each device's context, so it is set once per device.
    {
        static std::mutex mu;
        static std::vector<char> done;
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            std::lock_guard<std::mutex> lk(mu);
            if (static_cast<int>(done.size()) <= dev) done.resize(dev + 1, 0);
            if (!done[dev]) {
                (void)cudaFuncSetAttribute(sk_reduce_kernel,
                                           cudaFuncAttributePreferredSharedMemoryCarveout, 100);
                done[dev] = 1;
            }
        }
    }
    int chunks = reduce_chunks(bm, bn, a.sk_tiles, sms);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(a.sk_tiles) * chunks);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // Programmatic dependent launch: the reduction is scheduled as the main
    // kernel's CTAs finish and waits (griddepcontrol.wait) for its completion.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    GemmArgs args = a;
    void* params[] = {&args, &bm, &bn, &chunks};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&sk_reduce_kernel),
                                        params);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

}  // namespace sgemm
