// moba_decode.cu -- MoBA for one new query token per sequence against its
// KV cache (the newest token's k and v already written at position len - 1).
//
// Pages: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) sections 3.1
// and 4.1 (mean-pooled block keys, future blocks masked, top_k of the sorted
// block scores); "MOBA mixture of block attention for server-side long
// context" (hncyxsy.com/news/197418) section 3 (current block forced, causal
// inside it).  A decode step computes exactly the prefill forward's row
// i = len - 1 of each sequence.
//
// Two kernels, HBM-bound (one query row per (sequence, head) is a matrix-vector
// product, so CUDA cores):
//   decode_gate_kernel   one warp per (sequence, head): exact fp32 scores of
//                        the past blocks in the CUDA-core gate's summation
//                        order (lane l takes blocks l, l + 32, ...), the
//                        lanes' top lists merged by k-1 warp arg-max rounds;
//                        writes the selection (ascending, own block last).
//   decode_attn_kernel   one CTA per (sequence, head, selected block): four
//                        lanes per key (a quarter of the head dimension each),
//                        an online softmax per lane quad, the quads combined
//                        in shared memory into (max, sum, unnormalised O); the
//                        last CTA of a (sequence, head) (a ticket counter)
//                        merges the k partials by log-sum-exp into out, lse.
#include "moba.h"
#include "moba_internal.cuh"
#include "moba_ptx.cuh"
#include "moba_select.cuh"

namespace moba {
namespace dec {

constexpr int kGateWarps = 8;
constexpr int kAttnWarps = 4;
constexpr int kQuads = kAttnWarps * 8;  // keys in flight per CTA iteration

struct Args {
    const __nv_bfloat16 *q;       // [B][H][D]
    const __nv_bfloat16 *k, *v;   // [B][S_max][H][D]
    const float *kbar;            // [B * n_max][H][D]
    const int32_t *lens;          // [B], device
    __nv_bfloat16 *out;           // [B][H][D]
    float *lse;                   // [B][H]
    int32_t *idx;                 // [B][H][topk] or nullptr
    int32_t *sel;                 // [B][H][topk] scratch
    float *part_ml;               // [B][H][topk][2] scratch
    float *part_o;                // [B][H][topk][D] scratch
    int *ticket;                  // [B][H], zero on entry, zero again on exit
    int *status;
    int B, H, S_max, bs, topk, n_max;
    float scale_log2;
};

// the query's position, or -1 (recorded as an invalid argument) when the
// length is outside [1, S_max]
__device__ __forceinline__ int query_pos(const Args &a, int b) {
    const int len = __ldg(a.lens + b);
    if (len < 1 || len > a.S_max) {
        atomicCAS(a.status, 0, (int)MOBA_ERR_INVALID_ARG);
        return -1;
    }
    return len - 1;
}

template <int D, int KCAP>
__global__ void __launch_bounds__(32 * kGateWarps) decode_gate_kernel(Args a) {
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * kGateWarps + (threadIdx.x >> 5);
    if (w >= a.B * a.H) return;
    const int b = w / a.H, h = w % a.H;
    const int i = query_pos(a, b);
    const int km1 = a.topk - 1;
    int32_t *row = a.sel + (size_t)w * a.topk;
    if (i < 0) {
        if (lane == 0)
            for (int x = 0; x < a.topk; ++x) row[x] = -1;
        return;
    }
    const int ci = i / a.bs;
    int chosen[KCAP];  // selected past blocks, ascending (when scored)
    const bool scored = km1 > 0 && ci > km1;
    if (scored) {
        const __nv_bfloat16 *qg = a.q + (size_t)w * D;
        const float *kb_head = a.kbar + ((size_t)b * a.n_max * a.H + h) * D;
        float ts[KCAP];
        int ti[KCAP];
#pragma unroll
        for (int x = 0; x < KCAP; ++x) {
            ts[x] = -INFINITY;
            ti[x] = sel::kEmpty;
        }
        for (int c = lane; c < ci; c += 32)
            sel::top_insert<KCAP>(ts, ti, km1, sel::exact_score<D>(qg, kb_head + (size_t)c * a.H * D), c);
#pragma unroll
        for (int x = 0; x < KCAP; ++x) {
            chosen[x] = sel::kEmpty;
            if (x < km1) {
                float sv = ts[0];
                int cv = ti[0];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float s2 = __shfl_xor_sync(0xffffffffu, sv, o);
                    const int c2 = __shfl_xor_sync(0xffffffffu, cv, o);
                    if (s2 > sv || (s2 == sv && c2 < cv)) {
                        sv = s2;
                        cv = c2;
                    }
                }
                chosen[x] = cv;
                if (ti[0] == cv) {  // the winning lane drops its head
#pragma unroll
                    for (int y = 0; y + 1 < KCAP; ++y) {
                        ts[y] = ts[y + 1];
                        ti[y] = ti[y + 1];
                    }
                    ts[KCAP - 1] = -INFINITY;
                    ti[KCAP - 1] = sel::kEmpty;
                }
            }
        }
#pragma unroll
        for (int pass = 0; pass < KCAP; ++pass) {
#pragma unroll
            for (int x = pass & 1; x + 1 < KCAP; x += 2) {
                const int lo = min(chosen[x], chosen[x + 1]), hi = max(chosen[x], chosen[x + 1]);
                chosen[x] = lo;
                chosen[x + 1] = hi;
            }
        }
    }
    if (lane == 0) {
        // every past block when there are at most k-1 of them
        const int npast = scored ? km1 : min(ci, km1);
        if (scored) {
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x < npast) row[x] = chosen[x];
        } else {
            for (int x = 0; x < npast; ++x) row[x] = x;
        }
        row[npast] = ci;
        for (int x = npast + 1; x < a.topk; ++x) row[x] = -1;
        if (a.idx)
            for (int x = 0; x < a.topk; ++x) a.idx[(size_t)w * a.topk + x] = row[x];
    }
}

template <int D>
__global__ void __launch_bounds__(32 * kAttnWarps) decode_attn_kernel(Args a) {
    constexpr int DQ = D / 4;  // dims per lane of a quad
    __shared__ float s_m[kQuads], s_l[kQuads];
    __shared__ float s_o[kQuads][D + 4];
    __shared__ float s_scale[kQuads];
    __shared__ int s_last;
    const int bh = blockIdx.x, j = blockIdx.y;
    const int b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp * 8 + (lane >> 2), q4 = lane & 3;
    const int c = __ldg(a.sel + (size_t)bh * a.topk + j);
    const int i = (c >= 0) ? __ldg(a.lens + b) - 1 : -1;

    // the quad's running softmax over its keys (log2 domain)
    float m = -INFINITY, l = 0.f, o[DQ];
#pragma unroll
    for (int d = 0; d < DQ; ++d) o[d] = 0.f;
    if (c >= 0) {
        float qf[DQ];
        const __nv_bfloat16 *qp = a.q + (size_t)bh * D + q4 * DQ;
#pragma unroll
        for (int d8 = 0; d8 < DQ; d8 += 8) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(qp + d8));
            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(p2[e]);
                qf[d8 + 2 * e] = f.x;
                qf[d8 + 2 * e + 1] = f.y;
            }
        }
        const int t0 = c * a.bs, t1 = min(t0 + a.bs, i + 1);  // causal inside the own block
        const size_t tok_stride = (size_t)a.H * D;
        const __nv_bfloat16 *kbase = a.k + ((size_t)b * a.S_max * a.H + h) * D + q4 * DQ;
        const __nv_bfloat16 *vbase = a.v + ((size_t)b * a.S_max * a.H + h) * D + q4 * DQ;
        // Two keys per quad and iteration, their K and V loads all issued
        // before use.  The loop bound is the same for the whole warp (the
        // shuffles below need every lane); a quad past the block's end
        // computes nothing for that key.
        for (int t_base = t0; t_base < t1; t_base += 2 * kQuads) {
            int t[2];
            bool live[2];
            uint4 ku[2][DQ / 8], vu[2][DQ / 8];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                t[u] = t_base + u * kQuads + quad;
                live[u] = t[u] < t1;
#pragma unroll
                for (int x = 0; x < DQ / 8; ++x) {
                    ku[u][x] = live[u] ? __ldcs(reinterpret_cast<const uint4 *>(kbase + (size_t)t[u] * tok_stride) + x)
                                       : make_uint4(0, 0, 0, 0);
                    vu[u][x] = live[u] ? __ldcs(reinterpret_cast<const uint4 *>(vbase + (size_t)t[u] * tok_stride) + x)
                                       : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float s = 0.f;
#pragma unroll
                for (int x = 0; x < DQ / 8; ++x) {
                    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&ku[u][x]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(p2[e]);
                        s = fmaf(qf[8 * x + 2 * e], f.x, s);
                        s = fmaf(qf[8 * x + 2 * e + 1], f.y, s);
                    }
                }
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (!live[u]) continue;
                const float xl = s * a.scale_log2;
                const float m_new = fmaxf(m, xl);
                const float corr = ptx::fast_exp2(m - m_new);
                const float p = ptx::fast_exp2(xl - m_new);
                l = l * corr + p;
#pragma unroll
                for (int x = 0; x < DQ / 8; ++x) {
                    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&vu[u][x]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(p2[e]);
                        o[8 * x + 2 * e] = fmaf(p, f.x, o[8 * x + 2 * e] * corr);
                        o[8 * x + 2 * e + 1] = fmaf(p, f.y, o[8 * x + 2 * e + 1] * corr);
                    }
                }
                m = m_new;
            }
        }
    }
    // combine the quads: common max, rescaled sums and O
    if (q4 == 0) {
        s_m[quad] = m;
        s_l[quad] = l;
    }
    __syncthreads();
    if (tid == 0) {
        float M = -INFINITY;
        for (int x = 0; x < kQuads; ++x) M = fmaxf(M, s_m[x]);
        float L = 0.f;
        for (int x = 0; x < kQuads; ++x) {
            const float f = (s_m[x] == -INFINITY) ? 0.f : ptx::fast_exp2(s_m[x] - M);
            s_scale[x] = f;
            L += s_l[x] * f;
        }
        s_m[0] = M;
        s_l[0] = L;
    }
    __syncthreads();
    const float f = s_scale[quad];
#pragma unroll
    for (int d = 0; d < DQ; ++d) s_o[quad][q4 * DQ + d] = o[d] * f;
    __syncthreads();
    float *po = a.part_o + ((size_t)bh * a.topk + j) * D;
    for (int d = tid; d < D; d += 32 * kAttnWarps) {
        float acc = 0.f;
        for (int x = 0; x < kQuads; ++x) acc += s_o[x][d];
        po[d] = acc;
    }
    if (tid == 0) {
        a.part_ml[((size_t)bh * a.topk + j) * 2] = s_m[0];
        a.part_ml[((size_t)bh * a.topk + j) * 2 + 1] = s_l[0];
    }
    // the last CTA of this (sequence, head) merges the partials
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int t = atomicAdd(a.ticket + bh, 1);
        s_last = (t == a.topk - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const volatile float *pml = a.part_ml + (size_t)bh * a.topk * 2;
    float M = -INFINITY;
    for (int x = 0; x < a.topk; ++x)
        if (pml[2 * x + 1] > 0.f) M = fmaxf(M, pml[2 * x]);
    float L = 0.f;
    for (int x = 0; x < a.topk; ++x)
        if (pml[2 * x + 1] > 0.f) L += pml[2 * x + 1] * ptx::fast_exp2(pml[2 * x] - M);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const volatile float *pob = a.part_o + (size_t)bh * a.topk * D;
    for (int d = tid; d < D; d += 32 * kAttnWarps) {
        float acc = 0.f;
        for (int x = 0; x < a.topk; ++x)
            if (pml[2 * x + 1] > 0.f) acc += pob[(size_t)x * D + d] * ptx::fast_exp2(pml[2 * x] - M);
        a.out[(size_t)bh * D + d] = __float2bfloat16(acc * inv);
    }
    if (tid == 0) {
        a.lse[bh] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994530942f : -INFINITY;
        a.ticket[bh] = 0;  // ready for the next call
    }
}

}  // namespace dec

int decode_km1_max() { return 32; }

template <int D>
static cudaError_t launch_decode_d(const dec::Args &a, cudaStream_t st) {
    const int rows = a.B * a.H;
    const int km1 = a.topk - 1;
    const dim3 ggrid((rows + dec::kGateWarps - 1) / dec::kGateWarps);
#define MOBA_DEC_GATE(KC) \
    dec::decode_gate_kernel<D, KC><<<ggrid, 32 * dec::kGateWarps, 0, st>>>(a)
    if (km1 <= 1) MOBA_DEC_GATE(1);
    else if (km1 <= 2) MOBA_DEC_GATE(2);
    else if (km1 <= 4) MOBA_DEC_GATE(4);
    else if (km1 <= 8) MOBA_DEC_GATE(8);
    else if (km1 <= 16) MOBA_DEC_GATE(16);
    else MOBA_DEC_GATE(32);
#undef MOBA_DEC_GATE
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dec::decode_attn_kernel<D><<<dim3(rows, a.topk), 32 * dec::kAttnWarps, 0, st>>>(a);
    note_launches(2);
    return cudaGetLastError();
}

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *kbar,
                          const int32_t *lens, void *out, float *lse, int32_t *idx, int B, int H,
                          int S_max, int D, int bs, int topk, void *scratch, cudaStream_t st) {
    dec::Args a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k = static_cast<const __nv_bfloat16 *>(k);
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.kbar = kbar;
    a.lens = lens;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.idx = idx;
    a.B = B;
    a.H = H;
    a.S_max = S_max;
    a.bs = bs;
    a.topk = topk;
    a.n_max = (S_max + bs - 1) / bs;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    a.status = status_word();
    decode_scratch(scratch, B, H, D, topk, &a.sel, &a.part_ml, &a.part_o, &a.ticket);
    return D == 64 ? launch_decode_d<64>(a, st) : launch_decode_d<128>(a, st);
}

// scratch layout: selection, partial (max, sum), partial O, tickets
size_t decode_scratch(void *base, int B, int H, int D, int topk, int32_t **sel_, float **ml,
                      float **po, int **ticket) {
    const size_t rows = (size_t)B * H;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t b_sel = up(sizeof(int32_t) * rows * topk);
    const size_t b_ml = up(sizeof(float) * rows * topk * 2);
    const size_t b_o = up(sizeof(float) * rows * topk * D);
    const size_t b_t = up(sizeof(int) * rows);
    if (base) {
        char *p = static_cast<char *>(base);
        *sel_ = reinterpret_cast<int32_t *>(p);
        *ml = reinterpret_cast<float *>(p + b_sel);
        *po = reinterpret_cast<float *>(p + b_sel + b_ml);
        *ticket = reinterpret_cast<int *>(p + b_sel + b_ml + b_o);
    }
    return b_sel + b_ml + b_o + b_t;
}

size_t decode_ticket_offset(int B, int H, int D, int topk) {
    const size_t rows = (size_t)B * H;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    return up(sizeof(int32_t) * rows * topk) + up(sizeof(float) * rows * topk * 2) +
           up(sizeof(float) * rows * topk * D);
}

}  // namespace moba
