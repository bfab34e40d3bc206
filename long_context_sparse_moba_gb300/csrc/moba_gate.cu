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
#include <algorithm>

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
// S = max_len for every sequence).  Caller-provided offsets are checked first:
// they must start at 0, never decrease, give no sequence more than max_len
// tokens and end at `total`.  Offsets that fail leave every sequence empty,
// raise the `bad` flag that the later kernels test at entry, and record
// MOBA_ERR_INVALID_ARG in the device status word (moba_get_status): nothing
// is read or written through them.
// ---------------------------------------------------------------------------
__global__ void setup_kernel(const int *__restrict__ cu_in, int num_seqs, int S, int total, int bs,
                             int *__restrict__ cu, int *__restrict__ blk_base,
                             int *__restrict__ gtile, int *__restrict__ bad, int *status) {
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (cu_in) {
        for (int b = threadIdx.x; b <= num_seqs; b += blockDim.x) {
            const int x = cu_in[b];
            bool ok = (b > 0 || x == 0) && (b < num_seqs || x == total);
            if (b < num_seqs) {
                const int len = cu_in[b + 1] - x;
                ok = ok && len >= 0 && len <= S;
            }
            if (!ok) s_bad = 1;
        }
    }
    __syncthreads();
    const bool invalid = s_bad != 0;
    if (threadIdx.x == 0) {
        *bad = invalid ? 1 : 0;
        if (invalid && status) atomicCAS(status, 0, 1 /* MOBA_ERR_INVALID_ARG */);
    }
    auto len = [&](int b) { return invalid ? 0 : cu_in ? (cu_in[b + 1] - cu_in[b]) : S; };
    for (int b = threadIdx.x; b <= num_seqs; b += blockDim.x)
        cu[b] = invalid ? 0 : cu_in ? cu_in[b] : b * S;
    cta_exclusive_scan(
        num_seqs, [&](int b) { return (len(b) + bs - 1) / bs; },
        [&](int i, int v) { blk_base[i] = v; });
    cta_exclusive_scan(
        num_seqs, [&](int b) { return (len(b) + 127) / 128; },
        [&](int i, int v) { gtile[i] = v; });
}

cudaError_t launch_setup(const Plan &p, const int *cu_dev, Workspace &ws, cudaStream_t st) {
    setup_kernel<<<1, 1024, 0, st>>>(cu_dev, p.num_seqs, p.max_len, p.total, p.bs, ws.cu,
                                     ws.blk_base, ws.gtile, ws.bad, status_word());
    note_launches(1);
    return cudaGetLastError();
}

// idx rows of the paths that run no gate: the own block and every earlier
// block, ascending (top-1 keeps the own block alone), -1 padded
__global__ void fill_idx_kernel(Geometry g, int32_t *__restrict__ idx, int topk, int km1) {
    MOBA_RETURN_IF_BAD(g);
    const size_t R = (size_t)g.total * g.H;
    for (size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x; r < R;
         r += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(r / g.H);
        const int b = upper_index(g.cu, g.num_seqs, t);
        const int ci = (t - __ldg(g.cu + b)) / g.bs;
        const int npast = min(ci, km1);  // km1 = 0 for top-1, topk - 1 >= ci when dense
        int32_t *out = idx + r * topk;
        for (int x = 0; x < topk; ++x) out[x] = x < npast ? x : x == npast ? ci : -1;
    }
}

// ---------------------------------------------------------------------------
// K1: pool the keys of every block (mean, or with MAX the element-wise
// maximum: "MOBA mixture of block attention for server-side long context" §3
// allows either).  One CTA per (global block, group of
// 64 16-byte columns of the [H*D] token row).  Threads of a column walk the
// block's tokens with a stride of TG token groups; the TG partial sums are
// added (or maxed) in a fixed order, so the result is deterministic.  HBM-bound: every
// key byte is read once with 16-byte loads, coalesced along the token row.
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 256;

template <bool MAX>
__global__ __launch_bounds__(kPoolThreads) void kpool_kernel(Geometry g,
                                                              const __nv_bfloat16 *__restrict__ k,
                                                              float *__restrict__ kbar) {
    __shared__ float red[kPoolThreads][9];
    MOBA_RETURN_IF_BAD(g);
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
    // compensated (Kahan) fp32 sums: the mean of a 4096-token block stays
    // within ~1 ulp, which keeps the gate scores close to exact
    float acc[8], comp[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        acc[e] = MAX ? -INFINITY : 0.f;
        comp[e] = 0.f;
    }
    auto add8 = [&](const uint4 &u) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(p[e]);
            const float xs[2] = {f.x, f.y};
#pragma unroll
            for (int o = 0; o < 2; ++o) {
                const int k = 2 * e + o;
                if (MAX) {
                    acc[k] = fmaxf(acc[k], xs[o]);
                } else {
                    const float y = xs[o] - comp[k];
                    const float t = acc[k] + y;
                    comp[k] = (t - acc[k]) - y;
                    acc[k] = t;
                }
            }
        }
    };
    if (tg < TG && col < HD8) {
        const uint4 *base = reinterpret_cast<const uint4 *>(k) + col;
        const size_t row = (size_t)HD8;
        int t = t0 + tg;
        for (; t + 3 * TG < t1; t += 4 * TG) {
            uint4 u[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) u[j] = __ldcs(base + (size_t)(t + j * TG) * row);
#pragma unroll
            for (int j = 0; j < 4; ++j) add8(u[j]);
        }
        for (; t < t1; t += TG) add8(__ldcs(base + (size_t)t * row));
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
            for (int e = 0; e < 8; ++e) s[e] = MAX ? fmaxf(s[e], red[j * CW + colx][e]) : s[e] + red[j * CW + colx][e];
        const float cnt = MAX ? 1.f : (float)(t1 - t0);  // a max needs no division
        float4 *dst = reinterpret_cast<float4 *>(kbar + (size_t)gblk * g.H * g.D) + col * 2;
        dst[0] = make_float4(s[0] / cnt, s[1] / cnt, s[2] / cnt, s[3] / cnt);
        dst[1] = make_float4(s[4] / cnt, s[5] / cnt, s[6] / cnt, s[7] / cnt);
    }
}

// kbar -> (hi, lo) bf16 terms for the tensor-core gate, and the L2 norm of
// every pooled key; one warp per (block, head) row of D values
__global__ void kbar_split_kernel(const float *__restrict__ kbar, __nv_bfloat16 *__restrict__ hi,
                                  __nv_bfloat16 *__restrict__ lo, float *__restrict__ norm,
                                  int rows, int D) {
    const int lane = threadIdx.x & 31;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += (gridDim.x * blockDim.x) >> 5) {
        float ss = 0.f;
        for (int d = lane; d < D; d += 32) {
            const size_t i = (size_t)r * D + d;
            const float x = kbar[i];
            const __nv_bfloat16 h = __float2bfloat16_rn(x);
            hi[i] = h;
            lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
            ss = fmaf(x, x, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) norm[r] = sqrtf(ss);
    }
}

cudaError_t launch_kbar_split(const Plan &p, const float *kbar, __nv_bfloat16 *hi,
                              __nv_bfloat16 *lo, float *norm, cudaStream_t st) {
    const int rows = p.NBcap * p.H;
    const unsigned blocks = (unsigned)((rows + 7) / 8 < 8192 ? (rows + 7) / 8 : 8192);
    kbar_split_kernel<<<blocks, 256, 0, st>>>(kbar, hi, lo, norm, rows, p.D);
    note_launches(1);
    return cudaGetLastError();
}

static Geometry make_geo(const Plan &p, const Workspace &ws) {
    Geometry g;
    g.cu = ws.cu;
    g.blk_base = ws.blk_base;
    g.bad = ws.bad;
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
    if (p.pool == 1)
        kpool_kernel<true><<<grid, kPoolThreads, 0, st>>>(make_geo(p, ws), k, kbar);
    else
        kpool_kernel<false><<<grid, kPoolThreads, 0, st>>>(make_geo(p, ws), k, kbar);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K2 on the CUDA cores (selectable per call, and used when a
// sequence has more blocks than the tensor-core gate's TMEM holds): gate +
// top-k.  A CTA scores 128 consecutive query rows of one (sequence,
// head) against the pooled keys of that sequence's past blocks.  Four lanes
// share a row: lane j of a quad holds dims [j*D/4, (j+1)*D/4) of the quad's 4
// rows in fp32 registers, so every pooled-key load from shared memory feeds 16
// FMAs.  The quad adds its four partial dot products with two butterfly
// shuffles (all four lanes end with bit-identical sums) and lane j keeps the
// running top list of row j.  Pooled keys are staged 64 blocks at a time; the
// 16-byte chunks of a staged row are XOR-swizzled by the reading lane so the
// four distinct addresses of a load hit distinct banks.
// The top list keeps the KCAP best (score desc, block asc) candidates; blocks
// arrive in ascending order and a strictly greater score is needed to move
// ahead of an earlier block, which is the lower-index tie-break.  Rows whose
// own block has at most topk - 1 predecessors take them all without scoring.
// ---------------------------------------------------------------------------
constexpr int kGateThreads = 128;
constexpr int kGateRows = 128;
constexpr int kGateChunk = 64;
constexpr int kEmpty = 0x7fffffff;

template <int D, int KCAP>
__global__ __launch_bounds__(kGateThreads) void gate_kernel(
    Geometry g, const __nv_bfloat16 *__restrict__ q, const float *__restrict__ kbar,
    int32_t *__restrict__ idx, int topk) {
    constexpr int DL = D / 4;  // dims per lane
    constexpr int M = DL / 4;  // float4 chunks per lane
    __shared__ __align__(16) float skb[kGateChunk * D];
    __shared__ int s_cmax;
    MOBA_RETURN_IF_BAD(g);
    const int h = blockIdx.y, b = blockIdx.z, H = g.H;
    const int seq0 = __ldg(g.cu + b), L = __ldg(g.cu + b + 1) - seq0;
    const int i0 = blockIdx.x * kGateRows;
    if (i0 >= L) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = lane & 3, rbase = 32 * warp + 4 * (lane >> 2);
    const int km1 = topk - 1;
    const int bbase = __ldg(g.blk_base + b);

    const int my_i = i0 + rbase + j;
    const bool my_valid = my_i < L;
    const int my_ci = my_valid ? my_i / g.bs : 0;
    const int my_tok = seq0 + my_i;
    const bool my_scored = my_valid && km1 > 0 && my_ci > km1;

    if (tid == 0) s_cmax = 0;
    __syncthreads();
    if (my_scored) atomicMax(&s_cmax, my_ci);

    float qf[4][DL];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = i0 + rbase + r;
        const uint4 *qp = reinterpret_cast<const uint4 *>(q + ((size_t)(seq0 + i) * H + h) * D + j * DL);
#pragma unroll
        for (int c8 = 0; c8 < DL / 8; ++c8) {
            uint4 u = (i < L) ? __ldcs(qp + c8) : make_uint4(0, 0, 0, 0);
            const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = __bfloat1622float2(p2[e]);
                qf[r][8 * c8 + 2 * e] = f.x;
                qf[r][8 * c8 + 2 * e + 1] = f.y;
            }
        }
    }
    const int wneed = __reduce_max_sync(0xffffffffu, my_scored ? my_ci : 0);
    __syncthreads();
    const int cmax = s_cmax;

    float ts[KCAP];
    int ti[KCAP];
#pragma unroll
    for (int x = 0; x < KCAP; ++x) {
        ts[x] = -INFINITY;
        ti[x] = kEmpty;
    }
    const float *kb_head = kbar + ((size_t)bbase * H + h) * D;
    for (int c0 = 0; c0 < cmax; c0 += kGateChunk) {
        const int nrow = min(kGateChunk, cmax - c0);
        __syncthreads();
        for (int x = tid; x < nrow * (D / 4); x += kGateThreads) {
            const int row = x / (D / 4), ch = x % (D / 4);
            const int jj = ch / M, mm = ch % M;
            const float4 v = __ldg(reinterpret_cast<const float4 *>(kb_head + (size_t)(c0 + row) * H * D) + ch);
            reinterpret_cast<float4 *>(skb + row * D)[jj * M + (mm ^ jj)] = v;
        }
        __syncthreads();
        const int cend = min(c0 + kGateChunk, wneed);
        for (int c = c0; c < cend; ++c) {
            const float4 *kr = reinterpret_cast<const float4 *>(skb + (c - c0) * D) + j * M;
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float4 kv = kr[m ^ j];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    acc[r][0] = fmaf(qf[r][4 * m + 0], kv.x, acc[r][0]);
                    acc[r][1] = fmaf(qf[r][4 * m + 1], kv.y, acc[r][1]);
                    acc[r][2] = fmaf(qf[r][4 * m + 2], kv.z, acc[r][2]);
                    acc[r][3] = fmaf(qf[r][4 * m + 3], kv.w, acc[r][3]);
                }
            }
            float sc[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float x = (acc[r][0] + acc[r][1]) + (acc[r][2] + acc[r][3]);
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                sc[r] = x;
            }
            float cur = (j == 0) ? sc[0] : (j == 1) ? sc[1] : (j == 2) ? sc[2] : sc[3];
            if (my_scored && c < my_ci) {
                if (cur != cur) cur = -INFINITY;  // a NaN score ranks last
                int curi = c;
                bool ins = false;
#pragma unroll
                for (int x = 0; x < KCAP; ++x) {
                    // an empty slot takes any candidate, so all km1 slots fill
                    const bool take = (x < km1) && (ins || cur > ts[x] || ti[x] == kEmpty);
                    if (take) {
                        const float fs = ts[x];
                        const int fi = ti[x];
                        ts[x] = cur;
                        ti[x] = curi;
                        cur = fs;
                        curi = fi;
                        ins = true;
                    }
                }
            }
        }
    }

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
            npast = (km1 == 0) ? 0 : my_ci;  // every past block (my_ci <= km1)
#pragma unroll
            for (int x = 0; x < KCAP; ++x) ti[x] = x;
        }
        int32_t *out = idx + ((size_t)my_tok * H + h) * topk;
        if (my_scored) {
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x < npast) out[x] = ti[x];
        } else {
            for (int x = 0; x < npast; ++x) out[x] = x;  // npast may exceed KCAP here
        }
        out[npast] = my_ci;
        for (int x = npast + 1; x < topk; ++x) out[x] = -1;
    }
}

template <int D>
static void launch_gate_d(dim3 grid, cudaStream_t st, Geometry g, const __nv_bfloat16 *q,
                          const float *kbar, int32_t *idx, int topk) {
    const int km1 = topk - 1;
#define MOBA_GATE_CASE(KC)                                                        \
    gate_kernel<D, KC><<<grid, kGateThreads, 0, st>>>(g, q, kbar, idx, topk); \
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
                        const float *kbar, int32_t *idx, cudaStream_t st) {
    dim3 grid((p.max_len + kGateRows - 1) / kGateRows, p.H, p.num_seqs);
    Geometry g = make_geo(p, ws);
    if (p.D == 64) launch_gate_d<64>(grid, st, g, q, kbar, idx, p.topk);
    else launch_gate_d<128>(grid, st, g, q, kbar, idx, p.topk);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K3: regroup into per-(block, head) lists of the rows that selected that past
// block.  (a) count: every CTA histograms the selections of a contiguous range
// of rows in shared memory and adds the histogram into the global counts;
// (b) one CTA scans the counts into list and tile offsets (and the job table
// of the past-block attention); (c) scatter: every CTA histograms its rows
// again, reserves its range inside each list with one atomicSub per non-empty
// bin (which brings the counts back to zero) and writes each selection at its
// reserved position.  The order inside a list depends on which CTA reserved
// first; a row's result does not depend on which rows share its attention
// tile, so outputs stay deterministic.  With more bins than shared memory
// holds, every selection goes straight to the global counters.
// ---------------------------------------------------------------------------
constexpr int kRgThreads = 512;
constexpr int kRgSmemBins = 48 * 1024;  // 192 KB of shared-memory histogram at most

// Which own-block jobs are fused (job_nu[job] > 0); null when none is.  Job
// numbering of the own-block attention kernel: heads fastest, then sequences,
// then 256-row tiles from the last.
struct FusedJobs {
    const int *job_nu;
    int n_rtiles;
    __device__ __forceinline__ bool row_fused(const Geometry &g, int b, int i_loc, int h) const {
        if (!job_nu) return false;
        const int x = i_loc / kFuseRows;
        const int job = ((n_rtiles - 1 - x) * g.num_seqs + b) * g.H + h;
        return __ldg(job_nu + job) > 0;
    }
};

// calls f(bin, entry) for every past selection of row r = token * H + head
// (none for the rows of fused own-block jobs)
template <typename F>
__device__ __forceinline__ void for_each_selection(const Geometry &g, const int32_t *__restrict__ idx,
                                                   int topk, size_t r, const FusedJobs &fj, F f) {
    const int t = (int)(r / g.H), h = (int)(r % g.H);
    const int b = upper_index(g.cu, g.num_seqs, t);
    const int seq0 = __ldg(g.cu + b);
    const int ci = (t - seq0) / g.bs;
    if (fj.row_fused(g, b, t - seq0, h)) return;
    const int bbase = __ldg(g.blk_base + b);
    const int32_t *row = idx + r * topk;
    for (int s = 0; s < topk - 1; ++s) {
        const int c = __ldg(row + s);
        if (c < 0 || c >= ci) break;
        f((bbase + c) * g.H + h, (t << kSlotBits) | s);
    }
}

template <bool SMEM>
__global__ void __launch_bounds__(kRgThreads)
    regroup_count_kernel(Geometry g, const int32_t *__restrict__ idx, int topk, int rows_per_cta,
                         int N, int *__restrict__ counts, FusedJobs fj) {
    extern __shared__ int hist[];
    MOBA_RETURN_IF_BAD(g);
    const size_t R = (size_t)g.total * g.H;
    const size_t r0 = (size_t)blockIdx.x * rows_per_cta, r1 = min(R, r0 + rows_per_cta);
    if (SMEM) {
        for (int x = threadIdx.x; x < N; x += kRgThreads) hist[x] = 0;
        __syncthreads();
    }
    for (size_t r = r0 + threadIdx.x; r < r1; r += kRgThreads)
        for_each_selection(g, idx, topk, r, fj, [&](int bin, int) {
            if (SMEM) atomicAdd(&hist[bin], 1);
            else atomicAdd(counts + bin, 1);
        });
    if (SMEM) {
        __syncthreads();
        for (int x = threadIdx.x; x < N; x += kRgThreads)
            if (hist[x]) atomicAdd(counts + x, hist[x]);
    }
}

// After an earlier kernel has recorded an error in the device status word
// (a bounded wait gave up: the selection may be incomplete), the lists are
// published empty and the scatters write nothing, so that no later phase
// gathers through entries that were never written; the status stays set until
// the caller reads it.
__global__ void regroup_scan_kernel(const int *__restrict__ counts, int N, int tile_m,
                                    int *__restrict__ list_off, int *__restrict__ tile_off,
                                    int *__restrict__ job_list, const int *__restrict__ status) {
    const bool ok = status == nullptr || *(volatile const int *)status == 0;
    cta_exclusive_scan(
        N, [&](int i) { return ok ? counts[i] : 0; }, [&](int i, int v) { list_off[i] = v; });
    cta_exclusive_scan(
        N, [&](int i) { return ok ? (counts[i] + tile_m - 1) / tile_m : 0; },
        [&](int i, int v) {
            tile_off[i] = v;
            if (i < N && ok)  // the attention jobs of list i
                for (int t = 0, nt = (counts[i] + tile_m - 1) / tile_m; t < nt; ++t)
                    job_list[v + t] = i;
        });
}

template <bool SMEM>
__global__ void __launch_bounds__(kRgThreads)
    regroup_scatter_kernel(Geometry g, const int32_t *__restrict__ idx, int topk, int rows_per_cta,
                           int N, int *__restrict__ counts, const int *__restrict__ list_off,
                           int *__restrict__ list, FusedJobs fj, const int *__restrict__ status) {
    extern __shared__ int hist[];
    MOBA_RETURN_IF_BAD(g);
    if (status && *(volatile const int *)status != 0) return;  // the lists were published empty
    const size_t R = (size_t)g.total * g.H;
    const size_t r0 = (size_t)blockIdx.x * rows_per_cta, r1 = min(R, r0 + rows_per_cta);
    if (SMEM) {
        for (int x = threadIdx.x; x < N; x += kRgThreads) hist[x] = 0;
        __syncthreads();
        for (size_t r = r0 + threadIdx.x; r < r1; r += kRgThreads)
            for_each_selection(g, idx, topk, r, fj, [&](int bin, int) { atomicAdd(&hist[bin], 1); });
        __syncthreads();
        // this CTA's range in list x: [list_off + remaining - n, list_off + remaining);
        // a range that would start below the list (only when the counts and the
        // selection disagree) is refused whole: a negative start skips its writes
        for (int x = threadIdx.x; x < N; x += kRgThreads) {
            const int n = hist[x];
            if (n) {
                const int rem = atomicSub(counts + x, n);
                hist[x] = rem >= n ? __ldg(list_off + x) + rem - n : INT_MIN / 2;
            }
        }
        __syncthreads();
    }
    for (size_t r = r0 + threadIdx.x; r < r1; r += kRgThreads)
        for_each_selection(g, idx, topk, r, fj, [&](int bin, int entry) {
            // positions stay inside the list: ranges are reserved downwards from
            // its end and never below its start
            if (SMEM) {
                const int pos = atomicAdd(&hist[bin], 1);
                if (pos >= 0) list[pos] = entry;
            } else {
                const int rem = atomicSub(counts + bin, 1);
                if (rem > 0) list[__ldg(list_off + bin) + rem - 1] = entry;
            }
        });
}

cudaError_t launch_regroup(const Plan &p, const Workspace &ws, bool counted, bool skip_fused,
                           cudaStream_t st) {
    FusedJobs fj;
    fj.job_nu = skip_fused ? ws.job_nu : nullptr;
    fj.n_rtiles = (p.max_len + kFuseRows - 1) / kFuseRows;
    const int N = p.NBcap * p.H;
    const size_t R = (size_t)p.total * p.H;
    const bool smem = N <= kRgSmemBins;
    // enough rows per CTA that clearing and flushing the histogram stays cheap
    const int rows_per_cta = smem ? (int)std::max<long long>(2048, 2ll * N) : 4096;
    const unsigned grid = (unsigned)((R + rows_per_cta - 1) / rows_per_cta);
    const size_t hbytes = smem ? sizeof(int) * (size_t)N : 0;
    const Geometry g = make_geo(p, ws);
    cudaError_t e;
    if (smem) {
        e = cudaFuncSetAttribute(regroup_count_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hbytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(regroup_scatter_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hbytes);
        if (e != cudaSuccess) return e;
    }
    if (!counted) {
        if (smem)
            regroup_count_kernel<true><<<grid, kRgThreads, hbytes, st>>>(g, ws.idx, p.topk,
                                                                          rows_per_cta, N, ws.counts, fj);
        else
            regroup_count_kernel<false><<<grid, kRgThreads, 0, st>>>(g, ws.idx, p.topk,
                                                                     rows_per_cta, N, ws.counts, fj);
        note_launches(1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    regroup_scan_kernel<<<1, 1024, 0, st>>>(ws.counts, N, past_tile_rows(p), ws.list_off,
                                            ws.tile_off, ws.job_list, status_word());
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (smem)
        regroup_scatter_kernel<true><<<grid, kRgThreads, hbytes, st>>>(
            g, ws.idx, p.topk, rows_per_cta, N, ws.counts, ws.list_off, ws.list, fj, status_word());
    else
        regroup_scatter_kernel<false><<<grid, kRgThreads, 0, st>>>(
            g, ws.idx, p.topk, rows_per_cta, N, ws.counts, ws.list_off, ws.list, fj, status_word());
    note_launches(2);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The same lists in a fixed order (the backward's: it sums each key's dK and
// dV over its list tile by tile, so an order that changes from call to call
// changes their rounding).  Every CTA owns a range of whole tokens, all heads.
// (a) count: the CTA's histogram of its selections becomes its row of a
// [CTA][list] table; (b) a column scan turns every column into the CTAs'
// first positions inside that list (CTAs in token order) and its total into
// ws.counts; (c) the list and tile offsets as above; (d) scatter: warp w owns
// the heads h = w (mod 16) of its CTA -- so no other thread touches the lists
// of those heads -- and walks the CTA's tokens 32 at a time, slot by slot; the
// lanes that chose the same list take consecutive positions in lane order
// (__match_any_sync).  A list thus holds its entries ordered by CTA, 32-token
// group, slot and token, whatever the timing.
// ---------------------------------------------------------------------------
constexpr int kRgWarps = kRgThreads / 32;

// What the backward keeps beside each list entry: its row's forward lse (in
// log2 units) and delta; lse == nullptr when not asked for.
struct EntryMeta {
    const float *lse, *delta;  // lse [B][H][S] (fixed) or [H][total]; delta [H][total]
    int fixed, S_fixed;
    float *list_l2, *list_dl;
};

static int stable_tokens_per_cta(const Plan &p) {
    const long long N = (long long)p.NBcap * p.H;
    const long long rows = std::max<long long>(4096, 4 * N);  // as the histogram kernels above
    long long t = (rows + p.H - 1) / p.H;
    t = std::min<long long>(t, p.total);
    return (int)((t + 31) / 32 * 32);
}

int stable_regroup_ctas(const Plan &p) {
    const int tpc = stable_tokens_per_cta(p);
    return (p.total + tpc - 1) / tpc;
}

template <bool SMEM>
__global__ void __launch_bounds__(kRgThreads)
    regroup_count_cta_kernel(Geometry g, const int32_t *__restrict__ idx, int topk, int tpc, int N,
                             int *__restrict__ cta_hist) {
    extern __shared__ int hist[];
    MOBA_RETURN_IF_BAD(g);
    int *row = cta_hist + (size_t)blockIdx.x * N;  // zeroed beforehand without SMEM
    const size_t r0 = (size_t)blockIdx.x * tpc * g.H;
    const size_t r1 = min((size_t)g.total * g.H, r0 + (size_t)tpc * g.H);
    const FusedJobs none{nullptr, 0};
    if (SMEM) {
        for (int x = threadIdx.x; x < N; x += kRgThreads) hist[x] = 0;
        __syncthreads();
    }
    for (size_t r = r0 + threadIdx.x; r < r1; r += kRgThreads)
        for_each_selection(g, idx, topk, r, none, [&](int bin, int) {
            atomicAdd(SMEM ? &hist[bin] : row + bin, 1);
        });
    if (SMEM) {
        __syncthreads();
        for (int x = threadIdx.x; x < N; x += kRgThreads) row[x] = hist[x];
    }
}

// one thread per list: exclusive prefix of its column over the CTAs, total into counts
__global__ void regroup_colscan_kernel(int G, int N, int *__restrict__ cta_hist,
                                       int *__restrict__ counts) {
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= N) return;
    constexpr int kBatch = 8;  // loads in flight per thread
    int run = 0;
    for (int b0 = 0; b0 < G; b0 += kBatch) {
        int v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            v[u] = b0 + u < G ? cta_hist[(size_t)(b0 + u) * N + x] : 0;
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (b0 + u < G) {
                cta_hist[(size_t)(b0 + u) * N + x] = run;
                run += v[u];
            }
    }
    counts[x] = run;
}

template <bool SMEM>
__global__ void __launch_bounds__(kRgThreads)
    regroup_scatter_stable_kernel(Geometry g, const int32_t *__restrict__ idx, int topk, int tpc,
                                  int N, int *__restrict__ cta_hist,
                                  const int *__restrict__ list_off, int *__restrict__ list,
                                  const int *__restrict__ status, EntryMeta em) {
    extern __shared__ int hist[];
    MOBA_RETURN_IF_BAD(g);
    if (status && *(volatile const int *)status != 0) return;  // the lists were published empty
    int *row = cta_hist + (size_t)blockIdx.x * N;
    int *pos = SMEM ? hist : row;  // next free position of each list
    for (int x = threadIdx.x; x < N; x += kRgThreads) pos[x] = row[x] + __ldg(list_off + x);
    __syncthreads();
    const int t0 = blockIdx.x * tpc, t1 = min(g.total, t0 + tpc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    for (int h = warp; h < g.H; h += kRgWarps) {
        for (int tb = t0; tb < t1; tb += 32) {
            const int t = tb + lane;
            bool live = t < t1;
            int ci = 0, bbase = 0;
            float l2 = 0.f, dl = 0.f;  // my row's lse (log2) and delta, when asked for
            const int32_t *sel = idx;
            if (live) {
                const int b = upper_index(g.cu, g.num_seqs, t);
                const int seq0 = __ldg(g.cu + b);
                ci = (t - seq0) / g.bs;
                bbase = __ldg(g.blk_base + b);
                sel = idx + ((size_t)t * g.H + h) * topk;
                if (em.lse) {
                    const size_t li = em.fixed ? ((size_t)b * g.H + h) * em.S_fixed + (t - seq0)
                                               : (size_t)h * g.total + t;
                    l2 = __ldg(em.lse + li) * 1.4426950408889634f;
                    dl = __ldg(em.delta + (size_t)h * g.total + t);
                }
            }
            for (int s = 0; s < topk - 1; ++s) {
                const int c = live ? __ldg(sel + s) : -1;
                live = live && c >= 0 && c < ci;  // a row's selections end at its first invalid slot
                if (__ballot_sync(~0u, live) == 0u) break;
                const int bin = live ? (bbase + c) * g.H + h : -1;
                const unsigned peers = __match_any_sync(~0u, bin);
                const int base = live ? pos[bin] : 0;
                __syncwarp();
                if (live) {
                    const int at = base + __popc(peers & below);
                    list[at] = (t << kSlotBits) | s;
                    if (em.lse) {
                        em.list_l2[at] = l2;
                        em.list_dl[at] = dl;
                    }
                    if ((peers >> lane) == 1u) pos[bin] = base + __popc(peers);  // last of its group
                }
                __syncwarp();
            }
        }
    }
}

cudaError_t launch_regroup_stable(const Plan &p, const Workspace &ws, const float *lse,
                                  cudaStream_t st) {
    EntryMeta em{nullptr, nullptr, 0, 0, nullptr, nullptr};
    if (lse && ws.delta && ws.list_l2 && ws.list_dl)
        em = EntryMeta{lse, ws.delta, p.fixed ? 1 : 0, p.max_len, ws.list_l2, ws.list_dl};
    const int N = p.NBcap * p.H;
    const int tpc = stable_tokens_per_cta(p);
    const int G = stable_regroup_ctas(p);
    const bool smem = N <= kRgSmemBins;
    const size_t hbytes = smem ? sizeof(int) * (size_t)N : 0;
    const Geometry g = make_geo(p, ws);
    cudaError_t e;
    if (smem) {
        e = cudaFuncSetAttribute(regroup_count_cta_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hbytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(regroup_scatter_stable_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hbytes);
        if (e != cudaSuccess) return e;
        regroup_count_cta_kernel<true><<<G, kRgThreads, hbytes, st>>>(g, ws.idx, p.topk, tpc, N,
                                                                      ws.cta_hist);
    } else {
        if ((e = cudaMemsetAsync(ws.cta_hist, 0, sizeof(int) * (size_t)G * N, st)) != cudaSuccess)
            return e;
        regroup_count_cta_kernel<false><<<G, kRgThreads, 0, st>>>(g, ws.idx, p.topk, tpc, N,
                                                                  ws.cta_hist);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    regroup_colscan_kernel<<<(N + 255) / 256, 256, 0, st>>>(G, N, ws.cta_hist, ws.counts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    regroup_scan_kernel<<<1, 1024, 0, st>>>(ws.counts, N, past_tile_rows(p), ws.list_off,
                                            ws.tile_off, ws.job_list, status_word());
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (smem)
        regroup_scatter_stable_kernel<true><<<G, kRgThreads, hbytes, st>>>(
            g, ws.idx, p.topk, tpc, N, ws.cta_hist, ws.list_off, ws.list, status_word(), em);
    else
        regroup_scatter_stable_kernel<false><<<G, kRgThreads, 0, st>>>(
            g, ws.idx, p.topk, tpc, N, ws.cta_hist, ws.list_off, ws.list, status_word(), em);
    note_launches(4);
    return cudaGetLastError();
}

cudaError_t launch_fill_idx(const Plan &p, const Workspace &ws, int32_t *idx, cudaStream_t st) {
    const size_t R = (size_t)p.total * p.H;
    const unsigned blocks = (unsigned)std::min<size_t>((R + 255) / 256, 8192);
    fill_idx_kernel<<<blocks, 256, 0, st>>>(make_geo(p, ws), idx, p.topk, p.dense ? p.topk - 1 : p.km1);
    note_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Fusion test of each own-block job (256 rows of one block and head; block
// sizes a multiple of 256 keep a job inside one block, so its rows share one
// block index c > topk - 1).  The union of the rows' past selections has at
// most topk - 1 blocks exactly when every row selected the same topk - 1
// blocks.  Such a job is fused: the own-block kernel attends its rows to
// those blocks directly (no row does more work than on the block-major path)
// and its rows stay out of the regroup lists.  The rows of the first blocks
// (c <= topk - 1, which take every past block) are left to the lists, where
// they share long jobs with the rest of the sequence.  One warp per job
// compares every row's selection with the first row's and stops at the first
// difference.
// ---------------------------------------------------------------------------
constexpr int kUnionWarps = 8;

__global__ void __launch_bounds__(32 * kUnionWarps)
    union_kernel(Geometry g, const int32_t *__restrict__ idx, int topk, int n_rtiles,
                 int n_jobs, int *__restrict__ job_nu, int *__restrict__ job_ub,
                 int *__restrict__ counts, int *__restrict__ any_fused) {
    MOBA_RETURN_IF_BAD(g);
    const int job = blockIdx.x * kUnionWarps + (threadIdx.x >> 5);
    if (job >= n_jobs) return;  // whole warps leave together
    const int lane = threadIdx.x & 31, H = g.H, km1 = topk - 1;
    const int h = job % H, tt = job / H;
    const int b = tt % g.num_seqs;
    const int x = n_rtiles - 1 - tt / g.num_seqs;
    const int seq0 = __ldg(g.cu + b), L = __ldg(g.cu + b + 1) - seq0;
    const int r0 = x * kFuseRows;
    const int nrows = min(kFuseRows, L - r0);
    int nu = 0;
    int first[kMaxUnion];  // the first row's past blocks
#pragma unroll
    for (int s2 = 0; s2 < kMaxUnion; ++s2) first[s2] = -1;
    const int ci = r0 / g.bs;
    if (nrows > 0 && ci > km1) {
        const int32_t *row0 = idx + ((size_t)(seq0 + r0) * H + h) * topk;
#pragma unroll
        for (int s2 = 0; s2 < kMaxUnion; ++s2)
            if (s2 < km1) {
                const int c = __ldg(row0 + s2);
                if (c >= 0 && c < ci) first[s2] = c;
            }
        bool same = true;
        // warp-uniform trip count: every lane reaches each vote
        for (int base = 0; base < nrows; base += 32) {
            const int r = base + lane;
            if (r < nrows) {
                const int32_t *row = idx + ((size_t)(seq0 + r0 + r) * H + h) * topk;
#pragma unroll
                for (int s2 = 0; s2 < kMaxUnion; ++s2)
                    if (s2 < km1) {
                        int c = __ldg(row + s2);
                        if (c < 0 || c >= ci) c = -1;
                        same = same && c == first[s2];
                    }
            }
            if (!__all_sync(0xffffffffu, same)) break;
        }
        if (__all_sync(0xffffffffu, same)) {
#pragma unroll
            for (int s2 = 0; s2 < kMaxUnion; ++s2) nu += first[s2] >= 0;
        }
    }
    if (nu > 0 && lane < nu) {
        if (lane == 0) *any_fused = 1;
        if (counts) {
            // the job's selections leave the per-list counts the gate accumulated
            const int bbase = __ldg(g.blk_base + b);
            int c = -1;
#pragma unroll
            for (int s2 = 0; s2 < kMaxUnion; ++s2)
                if (s2 == lane) c = first[s2];
            atomicSub(counts + (size_t)(bbase + c) * H + h, nrows);
        }
    }
    if (lane == 0) job_nu[job] = nu;
    if (lane < kMaxUnion) {
        int c = -1;
#pragma unroll
        for (int s2 = 0; s2 < kMaxUnion; ++s2)
            if (s2 == lane) c = first[s2];
        job_ub[(size_t)job * kMaxUnion + lane] = lane < nu ? c : -1;
    }
}

bool fusion_enabled(const Plan &p) {
    return !p.dense && p.km1 > 0 && p.km1 <= kMaxUnion && p.bs % kFuseRows == 0 &&
           p.attn_kind == 0 && p.schedule == 0;
}



cudaError_t launch_union(const Plan &p, const Workspace &ws, bool counted, cudaStream_t st) {
    const int n_rtiles = (p.max_len + kFuseRows - 1) / kFuseRows;
    const long long jobs = (long long)n_rtiles * p.num_seqs * p.H;
    union_kernel<<<(unsigned)((jobs + kUnionWarps - 1) / kUnionWarps), 32 * kUnionWarps, 0, st>>>(
        make_geo(p, ws), ws.idx, p.topk, n_rtiles, (int)jobs, ws.job_nu,
        ws.job_ub, counted ? ws.counts : nullptr, ws.counts + (size_t)p.NBcap * p.H);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moba
