// The store of one 4-column chunk of C, shared by the FFMA kernels and the
// stream-K reduction.
//
// Plain form (the pages' epilogue-free store, "기존 작성한 GE_v2 의 regemm 타일드
// 커널의 1:1 매핑, gemm_tiled_test 작성", §6): C = acc.  Scaled form (the GE_v2
// kernel's epilogue that page's test kernel strips out, read with the usual BLAS
// conventions): C = alpha * acc + beta * C, where C is not read at all when
// beta == 0.  Columns gn .. gn+3 at or beyond N are not touched; the caller has
// already checked the row.
#pragma once

#include "sgemm_args.h"

namespace sgemm {

__device__ __forceinline__ float scale_one(const GemmArgs& a, float acc, const float* c) {
    return a.epi == kEpiAlphaBeta ? fmaf(a.alpha, acc, a.beta * *c) : a.alpha * acc;
}

__device__ __forceinline__ void store_c4(const GemmArgs& a, float* crow, int gn, float4 v) {
    const bool whole = a.c_vec && gn + 3 < a.N;
    if (a.epi != kEpiPlain) {
        if (a.epi == kEpiAlphaBeta && whole) {
            const float4 c = *reinterpret_cast<const float4*>(crow + gn);
            v = make_float4(fmaf(a.alpha, v.x, a.beta * c.x), fmaf(a.alpha, v.y, a.beta * c.y),
                            fmaf(a.alpha, v.z, a.beta * c.z), fmaf(a.alpha, v.w, a.beta * c.w));
        } else {
            if (gn + 0 < a.N) v.x = scale_one(a, v.x, crow + gn + 0);
            if (gn + 1 < a.N) v.y = scale_one(a, v.y, crow + gn + 1);
            if (gn + 2 < a.N) v.z = scale_one(a, v.z, crow + gn + 2);
            if (gn + 3 < a.N) v.w = scale_one(a, v.w, crow + gn + 3);
        }
    }
    if (whole) {
        *reinterpret_cast<float4*>(crow + gn) = v;
    } else {
        if (gn + 0 < a.N) crow[gn + 0] = v.x;
        if (gn + 1 < a.N) crow[gn + 1] = v.y;
        if (gn + 2 < a.N) crow[gn + 2] = v.z;
        if (gn + 3 < a.N) crow[gn + 3] = v.w;
    }
}

}  // namespace sgemm
