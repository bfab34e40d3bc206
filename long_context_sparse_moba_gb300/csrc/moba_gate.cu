// moba_gate.cu -- sequence tables, key pooling, gate + top-k and the regroup
// of queries by selected block.
//
// Pages: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) section 3.1
// (mean_pool block representation, future blocks masked) and section 4.1
// (sort block scores, keep top_k); "MOBA mixture of block attention for
// server-side long context" (hncyxsy.com/news/197418) section 3 (current block
// forced, inner product with the mean-pooled keys); "When a MoBA reproduction
// will not run" (mhpq.cn/news/582794) section 3.3 (the selected blocks of all
// queries are batched before attention -- here: a CSR list of query rows per
// (block, head)).
#include "moba_internal.cuh"

namespace moba {

// ---------------------------------------------------------------------------
// Single-CTA exclusive scan helper: out[i] = sum_{j<i} f(j), out[N] = total.
// ---------------------------------------------------------------------------
template <typename F, typename W>
__device__ void cta_exclusive_scan(int N, F f, W write) {
    __shared__ int warp_tot[32];
    __shared__ int carry;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) carry = 0;
    __syncthreads();
    const int per = (N + nt - 1) / nt;
    const int beg = min(tid * per, N), end = min(beg + per, N);
    int local = 0;
    for (int i = beg; i < end; ++i) local += f(i);
    // inclusive scan of `local` across the CTA
    int x = local;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = (lane < (nt >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    int run = x - local + (wid > 0 ? warp_tot[wid - 1] : 0);
    for (int i = beg; i < end; ++i) {
        write(i, run);
        run += f(i);
    }
    if (tid == nt - 1) write(N, run);
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Sequence tables.  cu_in: device int32 [num_seqs+1] or nullptr (fixed length
// S = max_len for every sequence).
// ---------------------------------------------------------------------------
__global__ void setup_kernel(const int *__restrict__ cu_in, int num_seqs, int S, int bs,
                             int *__restrict__ cu, int *__restrict__ blk_base) {
    auto len = [&](int b) { return cu_in ? (cu_in[b + 1] - cu_in[b]) : S; };
    for (int b = threadIdx.x; b <= num_seqs; b += blockDim.x)
        cu[b] = cu_in ? cu_in[b] : b * S;
    cta_exclusive_scan(
        num_seqs, [&](int b) { return (len(b) + bs - 1) / bs; },
        [&](int i, int v) { blk_base[i] = v; });
}

cudaError_t launch_setup(const Plan &p, const int *cu_dev, Workspace &ws, cudaStream_t st) {
    setup_kernel<<<1, 1024, 0, st>>>(cu_dev, p.num_seqs, p.max_len, p.bs, ws.cu, ws.blk_base);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K1: mean-pool the keys of every block.  One CTA per (global block, group of
// 64 16-byte columns of the [H*D] token row).  Threads of a column walk the
// block's tokens with a stride of TG token groups; the TG partial sums are
// added in a fixed order, so the result is deterministic.  HBM-bound: every
// key byte is read once with 16-byte loads, coalesced along the token row.
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 256;

__global__ __launch_bounds__(kPoolThreads) void kpool_kernel(Geometry g,
                                                              const __nv_bfloat16 *__restrict__ k,
                                                              float *__restrict__ kbar) {
    __shared__ float red[kPoolThreads][9];
    const int gblk = blockIdx.x;
    if (gblk >= __ldg(g.blk_base + g.num_seqs)) return;
    const int b = upper_index(g.blk_base, g.num_seqs, gblk);
    const int c = gblk - __ldg(g.blk_base + b);
    const int seq_end = __ldg(g.cu + b + 1);
    const int t0 = __ldg(g.cu + b) + c * g.bs;
    const int t1 = min(t0 + g.bs, seq_end);
    const int HD8 = g.H * g.D / 8;
    const int CW = min(HD8, 64);
    const int TG = kPoolThreads / CW;
    const int colx = threadIdx.x % CW, tg = threadIdx.x / CW;
    const int col = blockIdx.y * CW + colx;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    if (tg < TG && col < HD8) {
        const uint4 *base = reinterpret_cast<const uint4 *>(k) + col;
        const size_t row = (size_t)HD8;
        int t = t0 + tg;
        for (; t + 3 * TG < t1; t += 4 * TG) {
            uint4 u[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = __ldcs(base + (size_t)(t + j * TG) * row);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u[j]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = __bfloat1622float2(p[e]);
                    acc[2 * e] += f.x;
                    acc[2 * e + 1] += f.y;
                }
            }
        }
        for (; t < t1; t += TG) {
            uint4 u = __ldcs(base + (size_t)t * row);
            const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = __bfloat1622float2(p[e]);
                acc[2 * e] += f.x;
                acc[2 * e + 1] += f.y;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) red[threadIdx.x][e] = acc[e];
    __syncthreads();
    if (tg == 0 && col < HD8) {
        float s[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) s[e] = red[colx][e];
        for (int j = 1; j < TG; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[e] += red[j * CW + colx][e];
        const float cnt = (float)(t1 - t0);
        float4 *dst = reinterpret_cast<float4 *>(kbar + (size_t)gblk * g.H * g.D) + col * 2;
        dst[0] = make_float4(s[0] / cnt, s[1] / cnt, s[2] / cnt, s[3] / cnt);
        dst[1] = make_float4(s[4] / cnt, s[5] / cnt, s[6] / cnt, s[7] / cnt);
    }
}

static Geometry make_geo(const Plan &p, const Workspace &ws) {
    Geometry g;
    g.cu = ws.cu;
    g.blk_base = ws.blk_base;
    g.num_seqs = p.num_seqs;
    g.total = p.total;
    g.H = p.H;
    g.D = p.D;
    g.bs = p.bs;
    return g;
}

cudaError_t launch_kpool(const Plan &p, const Workspace &ws, const __nv_bfloat16 *k, float *kbar,
                         cudaStream_t st) {
    const int HD8 = p.H * p.D / 8;
    const int CW = HD8 < 64 ? HD8 : 64;
    dim3 grid(p.NBcap, (HD8 + CW - 1) / CW);
    kpool_kernel<<<grid, kPoolThreads, 0, st>>>(make_geo(p, ws), k, kbar);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K2: gate + top-k.  One thread per (token, head); a CTA holds 128
// consecutive tokens of one head, so the lanes of a warp read the same
// mean-pooled key (an L1 broadcast).  Scores are fp32 dot products with four
// interleaved partial sums.  The running top list keeps the KCAP best
// (score desc, block asc) candidates; since blocks are visited in ascending
// order, a strictly greater score is needed to move ahead of an earlier block,
// which gives the lower-index tie-break.  Rows whose own block has at most
// topk - 1 predecessors take them all without scoring.
// With COUNT, every past selection is also counted per (block, head) for the
// regroup.
// ---------------------------------------------------------------------------
constexpr int kGateThreads = 128;

template <int D, int KCAP, bool COUNT>
__global__ __launch_bounds__(kGateThreads) void gate_kernel(Geometry g,
                                                             const __nv_bfloat16 *__restrict__ q,
                                                             const float *__restrict__ kbar,
                                                             int32_t *__restrict__ idx, int topk,
                                                             int *__restrict__ counts) {
    const int h = blockIdx.y;
    const int t = blockIdx.x * kGateThreads + threadIdx.x;
    if (t >= g.total) return;
    const int H = g.H;
    const int b = upper_index(g.cu, g.num_seqs, t);
    const int i = t - __ldg(g.cu + b);
    const int ci = i / g.bs;
    const int km1 = topk - 1;
    const int bbase = __ldg(g.blk_base + b);
    int32_t *out = idx + ((size_t)t * H + h) * topk;

    if (km1 == 0) {  // top-1: the own block only
        out[0] = ci;
        return;
    }
    if (ci <= km1) {
        for (int j = 0; j < topk; ++j) out[j] = (j <= ci) ? j : -1;
        if (COUNT)
            for (int c = 0; c < ci; ++c) atomicAdd(counts + (size_t)(bbase + c) * H + h, 1);
        return;
    }

    float qf[D];
    {
        const uint4 *qp = reinterpret_cast<const uint4 *>(q + ((size_t)t * H + h) * D);
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            uint4 u = __ldcs(qp + j);
            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = __bfloat1622float2(p2[e]);
                qf[8 * j + 2 * e] = f.x;
                qf[8 * j + 2 * e + 1] = f.y;
            }
        }
    }
    float ts[KCAP];
    int ti[KCAP];
#pragma unroll
    for (int j = 0; j < KCAP; ++j) {
        ts[j] = -INFINITY;
        ti[j] = 0x7fffffff;
    }
    const float4 *kb = reinterpret_cast<const float4 *>(kbar + ((size_t)bbase * H + h) * D);
    const size_t kstride = (size_t)H * D / 4;
    for (int c = 0; c < ci; ++c) {
        const float4 *row = kb + (size_t)c * kstride;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < D / 4; ++j) {
            float4 m = __ldg(row + j);
            a0 = fmaf(qf[4 * j + 0], m.x, a0);
            a1 = fmaf(qf[4 * j + 1], m.y, a1);
            a2 = fmaf(qf[4 * j + 2], m.z, a2);
            a3 = fmaf(qf[4 * j + 3], m.w, a3);
        }
        float cur = (a0 + a1) + (a2 + a3);
        if (cur != cur) cur = -INFINITY;  // a NaN score ranks last
        int curi = c;
        bool ins = false;
#pragma unroll
        for (int j = 0; j < KCAP; ++j) {
            // an empty slot (index INT_MAX) takes any candidate, so every slot
            // is filled once km1 candidates have been seen
            bool take = (j < km1) && (ins || cur > ts[j] || ti[j] == 0x7fffffff);
            if (take) {
                float fs = ts[j];
                int fi = ti[j];
                ts[j] = cur;
                ti[j] = curi;
                cur = fs;
                curi = fi;
                ins = true;
            }
        }
    }
    // ascending block order (odd-even transposition sort; unused slots hold INT_MAX)
#pragma unroll
    for (int j = 0; j < KCAP; ++j)
        if (j >= km1) ti[j] = 0x7fffffff;
#pragma unroll
    for (int pass = 0; pass < KCAP; ++pass) {
#pragma unroll
        for (int j = pass & 1; j + 1 < KCAP; j += 2) {
            int lo = min(ti[j], ti[j + 1]), hi = max(ti[j], ti[j + 1]);
            ti[j] = lo;
            ti[j + 1] = hi;
        }
    }
#pragma unroll
    for (int j = 0; j < KCAP; ++j) {
        if (j < km1) {
            out[j] = ti[j];
            if (COUNT) atomicAdd(counts + (size_t)(bbase + ti[j]) * H + h, 1);
        }
    }
    out[km1] = ci;
}

template <int D, bool COUNT>
static void launch_gate_d(dim3 grid, cudaStream_t st, Geometry g, const __nv_bfloat16 *q,
                          const float *kbar, int32_t *idx, int topk, int *counts) {
    const int km1 = topk - 1;
#define MOBA_GATE_CASE(KC)                                                                     \
    gate_kernel<D, KC, COUNT><<<grid, kGateThreads, 0, st>>>(g, q, kbar, idx, topk, counts); \
    return;
    if (km1 <= 1) { MOBA_GATE_CASE(1) }
    if (km1 <= 2) { MOBA_GATE_CASE(2) }
    if (km1 <= 4) { MOBA_GATE_CASE(4) }
    if (km1 <= 8) { MOBA_GATE_CASE(8) }
    if (km1 <= 16) { MOBA_GATE_CASE(16) }
    MOBA_GATE_CASE(32)
#undef MOBA_GATE_CASE
}

cudaError_t launch_gate(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                        const float *kbar, int32_t *idx, bool count, cudaStream_t st) {
    dim3 grid((p.total + kGateThreads - 1) / kGateThreads, p.H);
    Geometry g = make_geo(p, ws);
    if (p.D == 64) {
        if (count) launch_gate_d<64, true>(grid, st, g, q, kbar, idx, p.topk, ws.counts);
        else launch_gate_d<64, false>(grid, st, g, q, kbar, idx, p.topk, nullptr);
    } else {
        if (count) launch_gate_d<128, true>(grid, st, g, q, kbar, idx, p.topk, ws.counts);
        else launch_gate_d<128, false>(grid, st, g, q, kbar, idx, p.topk, nullptr);
    }
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K3: regroup.  (a) one CTA scans the per-(block, head) counts into list and
// tile offsets; (b) every past selection is scattered into its list.  The
// order inside a list depends on atomic arrival; each row's result does not
// depend on which rows share its tile, so outputs stay deterministic.
// ---------------------------------------------------------------------------
__global__ void regroup_scan_kernel(const int *__restrict__ counts, int N, int tile_m,
                                    int *__restrict__ list_off, int *__restrict__ tile_off,
                                    int *__restrict__ cursor) {
    cta_exclusive_scan(
        N, [&](int i) { return counts[i]; },
        [&](int i, int v) {
            list_off[i] = v;
            if (i < N) cursor[i] = v;
        });
    cta_exclusive_scan(
        N, [&](int i) { return (counts[i] + tile_m - 1) / tile_m; },
        [&](int i, int v) { tile_off[i] = v; });
}

__global__ void regroup_scatter_kernel(Geometry g, const int32_t *__restrict__ idx, int topk,
                                       int *__restrict__ cursor, int *__restrict__ list) {
    const int h = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= g.total) return;
    const int b = upper_index(g.cu, g.num_seqs, t);
    const int ci = (t - __ldg(g.cu + b)) / g.bs;
    const int bbase = __ldg(g.blk_base + b);
    const int32_t *row = idx + ((size_t)t * g.H + h) * topk;
    for (int s = 0; s < topk - 1; ++s) {
        const int c = row[s];
        if (c < 0 || c >= ci) break;
        const int pos = atomicAdd(cursor + (size_t)(bbase + c) * g.H + h, 1);
        list[pos] = (t << kSlotBits) | s;
    }
}

int past_tile_rows();  // rows per tile of the past-block attention kernel

cudaError_t launch_regroup(const Plan &p, const Workspace &ws, cudaStream_t st) {
    const int N = p.NBcap * p.H;
    regroup_scan_kernel<<<1, 1024, 0, st>>>(ws.counts, N, past_tile_rows(), ws.list_off,
                                            ws.tile_off, ws.cursor);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 grid((p.total + 255) / 256, p.H);
    regroup_scatter_kernel<<<grid, 256, 0, st>>>(make_geo(p, ws), ws.idx, p.topk, ws.cursor,
                                                 ws.list);
    note_launches(2);
    return cudaGetLastError();
}

}  // namespace moba
