// moba_select.cuh -- the exact fp32 block score and the running top list,
// shared by the tensor-core gate's exact kernel and the decode gate so that
// both select exactly what the CUDA-core gate selects.
//
// Pages: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) sections 3.1
// and 4.1 (top_k of the sorted block scores); ties go to the lower block.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace moba {
namespace sel {

constexpr int kEmpty = 0x7fffffff;

// q_r . kbar_c in fp32 with the CUDA-core gate's order: lane partial j covers
// dims [j*D/4, (j+1)*D/4) with four interleaved FMA chains, then
// (p0 + p1) + (p2 + p3).
template <int D>
__device__ __noinline__ float exact_score(const __nv_bfloat16 *__restrict__ qg,
                                          const float *__restrict__ kb) {
    constexpr int DL = D / 4, M = DL / 4;
    float p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int d = j * DL + 4 * m;
            const uint2 qw = __ldg(reinterpret_cast<const uint2 *>(qg + d));
            const uint32_t lo = qw.x, hi = qw.y;
            const float4 k4 = __ldg(reinterpret_cast<const float4 *>(kb + d));
            const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lo));
            const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
            a0 = fmaf(q01.x, k4.x, a0);
            a1 = fmaf(q01.y, k4.y, a1);
            a2 = fmaf(q23.x, k4.z, a2);
            a3 = fmaf(q23.y, k4.w, a3);
        }
        p[j] = (a0 + a1) + (a2 + a3);
    }
    return (p[0] + p[1]) + (p[2] + p[3]);
}

// insert (x, c) into a descending list of km1 entries; equal scores keep the
// earlier (lower) block first; an empty slot takes any candidate
template <int KCAP>
__device__ __forceinline__ void top_insert(float (&ts)[KCAP], int (&ti)[KCAP], int km1, float x,
                                           int c) {
    if (x != x) x = -INFINITY;
    bool ins = false;
#pragma unroll
    for (int s = 0; s < KCAP; ++s) {
        const bool take = (s < km1) && (ins || x > ts[s] || ti[s] == kEmpty);
        if (take) {
            const float fs = ts[s];
            const int fi = ti[s];
            ts[s] = x;
            ti[s] = c;
            x = fs;
            c = fi;
            ins = true;
        }
    }
}

}  // namespace sel
}  // namespace moba
