// moba_gate_tc.cu -- gate + top-k with the block scores on the tensor cores.
//
// Pages: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) sections 3.1
// and 4.1 (mean-pooled block representation, future blocks masked, top_k of
// the sorted block scores); "MOBA mixture of block attention for
// server-side long context" (hncyxsy.com/news/197418) section 3 (current
// block forced; inner product with the mean-pooled keys).
//
// One CTA = 128 consecutive query rows of one (sequence, head), 128 threads;
// thread r owns row r.
//   1. TMA loads the rows' q (bf16) and the pooled keys of the sequence's
//      past blocks split into two bf16 terms, kbar ~= hi + lo (hi = bf16(kbar),
//      lo = bf16(kbar - hi)); one tcgen05.mma chain per 128 blocks computes
//      approx[r][c] = q_r . hi_c + q_r . lo_c into TMEM (fp32).
//   2. Each thread keeps the top (k-1) approximate scores of its row and the
//      threshold T (the (k-1)-th).  With |approx - exact| <= E, where
//      E = 2^-13 ||q_r|| max_c ||kbar_c|| (at least 8x the worst case of the
//      bf16 split, the fp32 MMA accumulation and the fp32 dot product), every
//      block the exact rule selects has approx >= T - 2E.
//   3. Only those candidates get the exact fp32 score, with the summation
//      order of the CUDA-core gate (four lane partials of four interleaved
//      sums), so the selection -- and its lower-index tie-break -- equals that
//      kernel's bit for bit.
// Rows whose own block has at most k-1 predecessors take them all.  With
// COUNT every past selection also gets its regroup ticket (shared-memory
// histogram + one global atomic per non-empty bin).
#include "moba.h"
#include "moba_internal.cuh"
#include "moba_ptx.cuh"

namespace moba {
namespace gate_tc {
using namespace ptx;

constexpr int kRows = 128;
constexpr int kThreads = 128;
constexpr int kMaxBlocks = 256;  // scored blocks a row may have (TMEM columns)
constexpr int kHistBins = 512;
constexpr int kEmpty = 0x7fffffff;

struct Args {
    Geometry g;
    const float *kbar;   // [NB][H][D] fp32
    const float *knorm;  // [NB][H] L2 norms of the pooled keys
    int32_t *idx;
    int *ticket;
    int *counts;
    int topk;
    int *status;
    long long wait_limit;
};

// CH = blocks per MMA chain (the MMA's N): 64 when every sequence has at most
// 64 blocks (a smaller footprint, three CTAs per SM), else 128
template <int D, int CH>
struct Smem {
    static constexpr int NB = D / 64;
    static constexpr uint32_t kQBox = 128 * 128;  // 128 rows x 128 bytes
    static constexpr uint32_t kBBox = CH * 128;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kHi = kQ + NB * kQBox;
    static constexpr uint32_t kLo = kHi + NB * kBBox;
    static constexpr uint32_t kTiles = kLo + NB * kBBox;
    static constexpr uint32_t kRequest = kTiles + 1024;
};

// bf16 element d of row r of a K-major, 128-byte-swizzled [128][D] tile
template <int D>
__device__ __forceinline__ uint32_t q_addr(uint32_t base, int r, int d) {
    const int box = d >> 6, dd = d & 63;
    return base + box * (128 * 128) + r * 128 + ((((dd >> 3) ^ (r & 7))) << 4) + (dd & 7) * 2;
}

// q_r . kbar_c in fp32 with the CUDA-core gate's order: lane partial j covers
// dims [j*D/4, (j+1)*D/4) with four interleaved FMA chains, then
// (p0 + p1) + (p2 + p3).
template <int D>
__device__ __forceinline__ float exact_score(uint32_t sq, int r, const float *__restrict__ kb) {
    constexpr int DL = D / 4, M = DL / 4;
    float p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int d = j * DL + 4 * m;
            uint32_t lo, hi;
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(q_addr<D>(sq, r, d)));
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

template <int D, int CH, int KCAP, bool COUNT>
__global__ void __launch_bounds__(kThreads)
    gate_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_hi,
                   const __grid_constant__ CUtensorMap tmap_lo, Args a) {
    using L = Smem<D, CH>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bars[2];  // loads, MMA chain
    __shared__ uint32_t tmem_slot;
    __shared__ int s_cmax, s_call, abort_word;
    __shared__ unsigned s_knmax;
    __shared__ int hist[kHistBins];
    const uint32_t raw = saddr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sQ = base + L::kQ, sHi = base + L::kHi, sLo = base + L::kLo;
    const uint32_t b_load = saddr(&bars[0]), b_mma = saddr(&bars[1]);

    const int h = blockIdx.y, b = blockIdx.z, H = a.g.H;
    const int seq0 = __ldg(a.g.cu + b), L_len = __ldg(a.g.cu + b + 1) - seq0;
    const int i0 = blockIdx.x * kRows;
    if (i0 >= L_len) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int km1 = a.topk - 1;
    const int bbase = __ldg(a.g.blk_base + b);
    const int my_i = i0 + tid;
    const bool my_valid = my_i < L_len;
    const int my_ci = my_valid ? my_i / a.g.bs : 0;
    const int my_tok = seq0 + my_i;
    const bool my_scored = my_valid && km1 > 0 && my_ci > km1;

    if (tid == 0) {
        s_cmax = 0;
        s_call = 0;
        s_knmax = 0u;
        abort_word = 0;
        mbar_init(b_load, 1);
        mbar_init(b_mma, 1);
        fence_mbar_init();
    }
    if (COUNT)
        for (int x = tid; x < kHistBins; x += kThreads) hist[x] = 0;
    __syncthreads();
    if (my_scored) atomicMax(&s_cmax, my_ci);
    if (my_valid) atomicMax(&s_call, my_ci);
    __syncthreads();
    const int cmax = s_cmax;  // blocks 0 .. cmax-1 are scored for some row
    Ctl ctl{reinterpret_cast<volatile int *>(&abort_word), a.status, a.wait_limit};

    float ts[KCAP];
    int ti[KCAP];
#pragma unroll
    for (int x = 0; x < KCAP; ++x) {
        ts[x] = -INFINITY;
        ti[x] = kEmpty;
    }
    bool ok = true;
    if (cmax > 0) {
        // TMEM: one fp32 column per scored block, rounded up to a power of 2
        const int nchunk = (cmax + CH - 1) / CH;
        const uint32_t tcols = (nchunk * CH <= 64) ? 64u : (nchunk * CH <= 128) ? 128u : 256u;
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             saddr(&tmem_slot)),
                         "r"(tcols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        // largest pooled-key norm among the scored blocks (for the margin)
        for (int c = tid; c < cmax; c += kThreads)
            atomicMax(&s_knmax, __float_as_uint(__ldg(a.knorm + (size_t)(bbase + c) * H + h)));
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = tmem_slot;
        constexpr uint32_t idesc = idesc_bf16(128, CH, 0);
        for (int ch = 0; ch < nchunk && ok; ++ch) {
            if (tid == 0) {
                const uint32_t bytes = (ch == 0 ? L::NB * L::kQBox : 0) + 2 * L::NB * L::kBBox;
                mbar_expect_tx(b_load, bytes);
                for (int x = 0; x < L::NB; ++x) {
                    if (ch == 0)
                        tma_load_3d(sQ + x * L::kQBox, &tmap_q, b_load, x * 64, h, seq0 + i0);
                    tma_load_3d(sHi + x * L::kBBox, &tmap_hi, b_load, x * 64, h, bbase + ch * CH);
                    tma_load_3d(sLo + x * L::kBBox, &tmap_lo, b_load, x * 64, h, bbase + ch * CH);
                }
                if (wait_bar(b_load, ch & 1, ctl)) {
                    tc_fence_after();
                    const uint32_t tS = tmem + ch * CH;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (uint32_t)(k % 4) * 32;
                        tc_mma(tS, sdesc(sQ + (k / 4) * L::kQBox + off, 16, 1024),
                               sdesc(sHi + (k / 4) * L::kBBox + off, 16, 1024), idesc, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (uint32_t)(k % 4) * 32;
                        tc_mma(tS, sdesc(sQ + (k / 4) * L::kQBox + off, 16, 1024),
                               sdesc(sLo + (k / 4) * L::kBBox + off, 16, 1024), idesc, 1u);
                    }
                    tc_commit(b_mma);
                }
            }
            // all threads: the chain finished (its B tiles may be overwritten)
            ok = __syncthreads_and(wait_bar(b_mma, ch & 1, ctl));
            tc_fence_after();
        }
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        if (ok) {
            // pass 1: top (k-1) of the approximate scores
            float as[KCAP];
            int ai[KCAP];
#pragma unroll
            for (int x = 0; x < KCAP; ++x) {
                as[x] = -INFINITY;
                ai[x] = kEmpty;
            }
            for (int c0 = 0; c0 < cmax; c0 += 32) {
                uint32_t v[32];
                tc_ld32(tmem + lane_off + c0, v);
                tc_wait_ld();
                if (my_scored) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c0 + e < my_ci) top_insert<KCAP>(as, ai, km1, __uint_as_float(v[e]), c0 + e);
                }
            }
            float T = -INFINITY;
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x == km1 - 1) T = as[x];
            // margin from the norms of q_r and of the pooled keys
            float qq = 0.f;
            if (my_scored)
#pragma unroll
                for (int d = 0; d < D; d += 8) {
                    uint32_t w[4];
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(q_addr<D>(sQ, tid, d)));
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                        qq = fmaf(f.x, f.x, fmaf(f.y, f.y, qq));
                    }
                }
            const float E = 0x1p-13f * sqrtf(qq) * __uint_as_float(s_knmax);
            const float thr = T - 2.f * E;
            // pass 2: exact fp32 scores of the candidates, in block order
            const float *kb_head = a.kbar + ((size_t)bbase * H + h) * D;
            for (int c0 = 0; c0 < cmax; c0 += 32) {
                uint32_t v[32];
                tc_ld32(tmem + lane_off + c0, v);
                tc_wait_ld();
                if (my_scored) {
                    uint32_t cand = 0u;  // bit e: block c0 + e is a candidate
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c0 + e < my_ci && __uint_as_float(v[e]) >= thr) cand |= 1u << e;
                    while (cand) {
                        const int c = c0 + __ffs(cand) - 1;
                        cand &= cand - 1;
                        top_insert<KCAP>(ts, ti, km1,
                                         exact_score<D>(sQ, tid, kb_head + (size_t)c * H * D), c);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(tcols)
                         : "memory");
        }
    }
    if (!ok) return;  // MOBA_ERR_TIMEOUT has been recorded

    // selected past blocks of my row, ascending
    int npast = 0;
    if (my_valid) {
        if (my_scored) {
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x >= km1) ti[x] = kEmpty;
#pragma unroll
            for (int pass = 0; pass < KCAP; ++pass) {
#pragma unroll
                for (int x = pass & 1; x + 1 < KCAP; x += 2) {
                    const int lo = min(ti[x], ti[x + 1]), hi = max(ti[x], ti[x + 1]);
                    ti[x] = lo;
                    ti[x + 1] = hi;
                }
            }
            npast = km1;
        } else {
            npast = (km1 == 0) ? 0 : my_ci;
#pragma unroll
            for (int x = 0; x < KCAP; ++x) ti[x] = x;
        }
        int32_t *out = a.idx + ((size_t)my_tok * H + h) * a.topk;
        if (my_scored) {
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x < npast) out[x] = ti[x];
        } else {
            for (int x = 0; x < npast; ++x) out[x] = x;
        }
        out[npast] = my_ci;
        for (int x = npast + 1; x < a.topk; ++x) out[x] = -1;
    }
    if (COUNT) {
        int rank[KCAP];
#pragma unroll
        for (int x = 0; x < KCAP; ++x) {
            rank[x] = 0;
            if (x < npast) {
                const int c = ti[x];
                rank[x] = (c < kHistBins) ? atomicAdd(&hist[c], 1)
                                          : atomicAdd(a.counts + (size_t)(bbase + c) * H + h, 1);
            }
        }
        __syncthreads();
        const int nbins = min(kHistBins, s_call);
        for (int x = tid; x < nbins; x += kThreads) {
            const int n = hist[x];
            hist[x] = n ? atomicAdd(a.counts + (size_t)(bbase + x) * H + h, n) : 0;
        }
        __syncthreads();
        if (my_valid) {
            int *tk = a.ticket + ((size_t)my_tok * H + h) * km1;
#pragma unroll
            for (int x = 0; x < KCAP; ++x) {
                if (x < npast) {
                    const int c = ti[x];
                    tk[x] = (c < kHistBins) ? hist[c] + rank[x] : rank[x];
                }
            }
        }
    }
}

}  // namespace gate_tc

bool gate_tc_supported(const Plan &p) {
    // TMEM holds two chunks of 128 block scores; the exact pass keeps the
    // top list in registers
    const long long nmax = (p.max_len + p.bs - 1) / p.bs;
    return nmax <= gate_tc::kMaxBlocks && p.topk - 1 <= 32 && (p.D == 64 || p.D == 128);
}

template <int D, int CH, bool COUNT>
static cudaError_t launch_gate_tc_d(const Plan &p, const gate_tc::Args &a, const __nv_bfloat16 *q,
                                    const __nv_bfloat16 *khi, const __nv_bfloat16 *klo,
                                    cudaStream_t st) {
    CUtensorMap mq, mh, ml;
    if (!make_tma_3d(&mq, q, p.total, p.H, D, 128) || !make_tma_3d(&mh, khi, p.NBcap, p.H, D, CH) ||
        !make_tma_3d(&ml, klo, p.NBcap, p.H, D, CH))
        return cudaErrorInvalidValue;
    dim3 grid((p.max_len + gate_tc::kRows - 1) / gate_tc::kRows, p.H, p.num_seqs);
    const int smem = gate_tc::Smem<D, CH>::kRequest;
    const int km1 = p.topk - 1;
#define MOBA_GATE_TC_CASE(KC)                                                                 \
    {                                                                                         \
        auto kern = gate_tc::gate_tc_kernel<D, CH, KC, COUNT>;                                    \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             smem);                                           \
        if (e != cudaSuccess) return e;                                                       \
        kern<<<grid, gate_tc::kThreads, smem, st>>>(mq, mh, ml, a);                           \
        return cudaGetLastError();                                                            \
    }
    if (km1 <= 1) MOBA_GATE_TC_CASE(1)
    if (km1 <= 2) MOBA_GATE_TC_CASE(2)
    if (km1 <= 4) MOBA_GATE_TC_CASE(4)
    if (km1 <= 8) MOBA_GATE_TC_CASE(8)
    if (km1 <= 16) MOBA_GATE_TC_CASE(16)
    MOBA_GATE_TC_CASE(32)
#undef MOBA_GATE_TC_CASE
}

cudaError_t launch_gate_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                           const float *kbar, const __nv_bfloat16 *khi, const __nv_bfloat16 *klo,
                           const float *knorm, int32_t *idx, bool count, cudaStream_t st) {
    gate_tc::Args a;
    a.g.cu = ws.cu;
    a.g.blk_base = ws.blk_base;
    a.g.num_seqs = p.num_seqs;
    a.g.total = p.total;
    a.g.H = p.H;
    a.g.D = p.D;
    a.g.bs = p.bs;
    a.kbar = kbar;
    a.knorm = knorm;
    a.idx = idx;
    a.ticket = count ? ws.ticket : nullptr;
    a.counts = count ? ws.counts : nullptr;
    a.topk = p.topk;
    a.status = status_word();
    a.wait_limit = tc_wait_limit();
    const bool small = (p.max_len + p.bs - 1) / p.bs <= 64;
    cudaError_t e;
#define MOBA_GATE_TC_D(DD, CC)                                                  \
    e = count ? launch_gate_tc_d<DD, CC, true>(p, a, q, khi, klo, st)          \
              : launch_gate_tc_d<DD, CC, false>(p, a, q, khi, klo, st);
    if (p.D == 64) {
        if (small) { MOBA_GATE_TC_D(64, 64) } else { MOBA_GATE_TC_D(64, 128) }
    } else {
        if (small) { MOBA_GATE_TC_D(128, 64) } else { MOBA_GATE_TC_D(128, 128) }
    }
#undef MOBA_GATE_TC_D
    note_launches(1);
    return e;
}

}  // namespace moba
