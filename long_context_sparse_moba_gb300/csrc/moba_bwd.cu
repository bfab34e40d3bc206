// moba_bwd.cu -- backward pass of MoBA attention: dq, dk, dv through the
// selected blocks, with the gate's selection held fixed (top-k is piecewise
// constant and passes no gradient; none reaches the pooled keys).
//
// Page: "MOBA mixture of block attention for server-side long context"
// (hncyxsy.com/news/197418) section 3 trains MoBA layers end to end and
// attributes a higher SFT loss to the sparse gradient path; the selection and
// the attention being differentiated are those of the forward pass
// ("Moonshot MoBA paper explained", gsyq.cn/news/227272, sections 3.1, 4.1).
//
// For row i with selected keys J_i (its own block up to i, and every key of
// its selected past blocks), P_ij = exp(s_ij / sqrt(D) - lse_i),
// delta_i = dO_i . O_i and dS_ij = P_ij (dO_i . v_j - delta_i):
//   dq_i = sum_j dS_ij k_j / sqrt(D),  dk_j = sum_i dS_ij q_i / sqrt(D),
//   dv_j = sum_i P_ij dO_i.
//
// Three kernels:
//   bwd_delta_kernel  -- delta = rowwise dO . O (a warp per (token, head));
//   bwd_kv_kernel     -- key-major: one work unit = 64 keys of one block of
//                        one head.  It walks every query row that attends to
//                        those keys -- the rows of the block itself from the
//                        unit's first key on (causal mask on the diagonal;
//                        on the dense path every later row of the sequence)
//                        and the rows of later blocks that selected the block
//                        (the regroup list of the forward pass) -- in tiles
//                        of 64, and per tile forms S^T = K Q^T and
//                        dP^T = V dO^T on the tensor cores (mma.sync bf16,
//                        fp32 accumulate), P and dS in fp32, then
//                        dV += P^T dO, dK += dS^T Q (registers, written once
//                        per unit: every key belongs to exactly one unit) and
//                        dQ += dS K added into an fp32 accumulator with
//                        16-byte vector atomics; the next tile's rows load
//                        while the dQ products run;
//   bwd_dq_kernel     -- dq = bf16(accumulator / sqrt(D)).
// 8 warps: for S^T and dP^T warp w takes keys 16 (w % 4) .. +15 x query rows
// 32 (w / 4) .. +31; for dV and dK keys 16 (w % 4) .. +15 x the column half
// w / 4 of D; for dQ query rows 16 (w % 4) .. +15 x the same column half.
// P^T, dS^T and dS pass between the phases through shared memory (bf16).
#include <algorithm>

#include "moba_internal.cuh"
#include "moba_mma.cuh"

namespace moba {

namespace bwd {

using namespace mma;

constexpr int kM = 64;          // query rows per tile
constexpr int kN = 64;          // keys per work unit
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
    Geometry g;
    const __nv_bfloat16 *q, *k, *v, *dout;
    const float *lse;           // forward lse, natural log, forward layout
    const float *delta;         // [H][total]
    float *dq_acc;              // [total][H][D], zero on entry
    __nv_bfloat16 *dq_out, *dk, *dv;  // [total][H][D]
    int fixed, S_fixed, dense, km1;
    const int *list, *list_off; // regroup lists (past selections)
    int tiles_per_block;        // bs / kN
    long long n_units;          // NBcap * H * tiles_per_block
    float scale, scale_log2;
};

template <int D>
constexpr int smem_bytes() {
    return 2 * kN * D * 2 + 2 * kM * D * 2 + 3 * kN * kM * 2 + 2 * 3 * kM * 4;
}

// 64 rows x D of a token-gathered bf16 matrix into a swizzled tile; rows with
// token < 0 are zero-filled (source size 0; the address stays valid).
template <int D, typename TokOf>
__device__ __forceinline__ void load_rows(uint32_t s_base, const __nv_bfloat16 *base,
                                          size_t rstride, TokOf tok_of) {
    constexpr int CH = D / 8;
#pragma unroll
    for (int j = 0; j < (64 * CH) / kThreads; ++j) {
        const int id = threadIdx.x + j * kThreads;
        const int r = id / CH, ch = id % CH;
        const int tok = tok_of(r);
        const __nv_bfloat16 *src = tok >= 0 ? base + (size_t)tok * rstride + ch * 8 : base;
        cp_async16(s_base + swz<D>(r, ch), src, tok >= 0);
    }
}

// delta = dO . O per (token, head) row: D / 8 lanes per row, 16 bytes of each
// tensor per lane, four row groups of the warp in flight per pass
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16 *__restrict__ out,
                                                        const __nv_bfloat16 *__restrict__ dout,
                                                        float *__restrict__ delta,
                                                        long long rows, int H, int total) {
    constexpr int LPR = D / 8;       // lanes per row
    constexpr int RPW = 32 / LPR;    // rows per warp and pass
    constexpr int U = 4;             // passes in flight
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const long long warps = (long long)gridDim.x * 8;
    for (long long r0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW * U; r0 < rows;
         r0 += warps * RPW * U) {
        uint4 x[U], y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long r = r0 + u * RPW + sub;
            if (r < rows) {
                x[u] = __ldg(reinterpret_cast<const uint4 *>(out + r * D) + li);
                y[u] = __ldg(reinterpret_cast<const uint4 *>(dout + r * D) + li);
            } else {
                x[u] = y[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const __nv_bfloat162 *xa = reinterpret_cast<const __nv_bfloat162 *>(&x[u]);
            const __nv_bfloat162 *ya = reinterpret_cast<const __nv_bfloat162 *>(&y[u]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a2 = __bfloat1622float2(xa[e]), b2 = __bfloat1622float2(ya[e]);
                acc = fmaf(a2.x, b2.x, fmaf(a2.y, b2.y, acc));
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const long long r = r0 + u * RPW + sub;
            // [H][total]: each head's rows contiguous
            if (li == 0 && r < rows) delta[(size_t)(r % H) * total + r / H] = acc;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) bwd_kv_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int KS = D / 16;   // k-steps over the head dimension
    constexpr int NH = D / 16;   // 8-column tiles in a warp's half of D
    uint8_t *pK = smem;
    uint8_t *pV = pK + kN * D * 2;
    uint8_t *pQ = pV + kN * D * 2;
    uint8_t *pO = pQ + kM * D * 2;
    uint8_t *pP = pO + kM * D * 2;   // P^T  [key][row]
    uint8_t *pS = pP + kN * kM * 2;  // dS^T [key][row]
    uint8_t *pR = pS + kN * kM * 2;  // dS   [row][key]
    // per-row metadata of two query tiles (the current and the next)
    int *r_tok = reinterpret_cast<int *>(pR + kM * kN * 2);
    float *r_lse = reinterpret_cast<float *>(r_tok + 2 * kM);  // log2 domain
    float *r_del = r_lse + 2 * kM;
    const uint32_t sK = smem_u32(pK), sV = smem_u32(pV), sQ = smem_u32(pQ), sO = smem_u32(pO);
    const uint32_t sP = smem_u32(pP), sS = smem_u32(pS), sR = smem_u32(pR);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wm = warp & 3, wn = warp >> 2;
    const int g = lane >> 2, t = lane & 3;
    const int H = a.g.H;
    MOBA_RETURN_IF_BAD(a.g);
    const size_t rstride = (size_t)H * D;
    const int NB = __ldg(a.g.blk_base + a.g.num_seqs);

    for (long long u = blockIdx.x; u < a.n_units; u += gridDim.x) {
        const int kt = (int)(u % a.tiles_per_block);
        const long long L = u / a.tiles_per_block;
        const int gblk = (int)(L / H), h = (int)(L % H);
        if (gblk >= NB) break;  // units run in block order: the rest are past the end too
        const int b = upper_index(a.g.blk_base, a.g.num_seqs, gblk);
        const int c = gblk - __ldg(a.g.blk_base + b);
        const int seq0 = __ldg(a.g.cu + b), seq_end = __ldg(a.g.cu + b + 1);
        const int kv0 = seq0 + c * a.g.bs;
        const int kv_end = min(kv0 + a.g.bs, seq_end);
        const int key0 = kv0 + kt * kN;
        if (key0 >= kv_end) continue;
        const int nkeys = min(kN, kv_end - key0);
        const int own_end = a.dense ? seq_end : kv_end;
        const int n_own = (own_end - key0 + kM - 1) / kM;
        int lbeg = 0, lcnt = 0;
        if (!a.dense && a.km1 > 0) {
            lbeg = __ldg(a.list_off + L);
            lcnt = __ldg(a.list_off + L + 1) - lbeg;
        }
        const int n_tiles = n_own + (lcnt + kM - 1) / kM;

        // token of row r of query tile qt (-1: no row)
        auto tok_of = [&](int qt, int r) -> int {
            if (qt < n_own) {
                const int x = key0 + qt * kM + r;
                return x < own_end ? x : -1;
            }
            const int pr = (qt - n_own) * kM + r;
            return pr < lcnt ? (__ldg(a.list + lbeg + pr) >> kSlotBits) : -1;
        };
        // row token, lse (log2) and delta of tile qt into metadata buffer mb
        auto fill_meta = [&](int qt, int mb) {
            if (threadIdx.x < kM) {
                const int r = threadIdx.x;
                const int tok = tok_of(qt, r);
                float l2 = 0.f, dl = 0.f;
                if (tok >= 0) {
                    const size_t li = a.fixed ? ((size_t)b * H + h) * a.S_fixed + (tok - seq0)
                                              : (size_t)h * a.g.total + tok;
                    l2 = __ldg(a.lse + li) * kLog2e;
                    dl = __ldg(a.delta + (size_t)h * a.g.total + tok);
                }
                r_tok[mb * kM + r] = tok;
                r_lse[mb * kM + r] = l2;
                r_del[mb * kM + r] = dl;
            }
        };

        load_rows<D>(sK, a.k + (size_t)h * D, rstride,
                     [&](int r) { return r < nkeys ? key0 + r : -1; });
        load_rows<D>(sV, a.v + (size_t)h * D, rstride,
                     [&](int r) { return r < nkeys ? key0 + r : -1; });
        load_rows<D>(sQ, a.q + (size_t)h * D, rstride, [&](int r) { return tok_of(0, r); });
        load_rows<D>(sO, a.dout + (size_t)h * D, rstride, [&](int r) { return tok_of(0, r); });
        cp_async_commit();
        fill_meta(0, 0);

        float dk[NH][4], dv[NH][4];
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) dk[j][e] = dv[j][e] = 0.f;

        // Per tile: [wait for Q, dO] S^T, dP^T -> P, dS [sync] dV, dK [sync]
        // start loading the next tile's Q, dO, then dQ and its atomics.
        for (int qt = 0; qt < n_tiles; ++qt) {
            const bool own = qt < n_own;
            const int *m_tok = r_tok + (qt & 1) * kM;
            const float *m_lse = r_lse + (qt & 1) * kM;
            const float *m_del = r_del + (qt & 1) * kM;
            cp_async_wait<0>();
            __syncthreads();

            // S^T and dP^T: keys 16 wm .. +15 x rows 32 wn .. +31
            float s[4][4], dp[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[j][e] = dp[j][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t ka[4], va[4];
                const uint32_t aoff = swz<D>(wm * 16 + (lane & 15), ks * 2 + (lane >> 4));
                ldsm_x4(ka[0], ka[1], ka[2], ka[3], sK + aoff);
                ldsm_x4(va[0], va[1], va[2], va[3], sV + aoff);
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    const uint32_t boff = swz<D>(wn * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3),
                                                 ks * 2 + ((lane >> 3) & 1));
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(b0, b1, b2, b3, sQ + boff);
                    mma16816(s[2 * np], ka, b0, b1);
                    mma16816(s[2 * np + 1], ka, b2, b3);
                    ldsm_x4(b0, b1, b2, b3, sO + boff);
                    mma16816(dp[2 * np], va, b0, b1);
                    mma16816(dp[2 * np + 1], va, b2, b3);
                }
            }
            // P, dS (fp32) -> bf16 tiles in shared memory
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int kl = wm * 16 + g + 8 * hh;
                    const int rl = wn * 32 + 8 * j + 2 * t;
                    float pv[2], dsv[2];
#pragma unroll
                    for (int e1 = 0; e1 < 2; ++e1) {
                        const int e = hh * 2 + e1;
                        const int r = rl + e1;
                        const int tok = m_tok[r];
                        const bool ok = tok >= 0 && kl < nkeys && (!own || key0 + kl <= tok);
                        const float p = ok ? fast_exp2(s[j][e] * a.scale_log2 - m_lse[r]) : 0.f;
                        pv[e1] = p;
                        dsv[e1] = p * (dp[j][e] - m_del[r]);
                    }
                    const uint32_t o_kr = swz<64>(kl, rl >> 3) + (rl & 7) * 2;
                    *reinterpret_cast<uint32_t *>(pP + o_kr) = pack_bf16(pv[0], pv[1]);
                    *reinterpret_cast<uint32_t *>(pS + o_kr) = pack_bf16(dsv[0], dsv[1]);
                    *reinterpret_cast<__nv_bfloat16 *>(pR + swz<64>(rl, kl >> 3) + (kl & 7) * 2) =
                        __float2bfloat16_rn(dsv[0]);
                    *reinterpret_cast<__nv_bfloat16 *>(pR + swz<64>(rl + 1, kl >> 3) + (kl & 7) * 2) =
                        __float2bfloat16_rn(dsv[1]);
                }
            }
            __syncthreads();

            // dV += P^T dO, dK += dS^T Q: keys 16 wm .. +15 x column half wn
#pragma unroll
            for (int ks = 0; ks < kM / 16; ++ks) {
                uint32_t pa[4], sa[4];
                const uint32_t aoff = swz<64>(wm * 16 + (lane & 15), ks * 2 + (lane >> 4));
                ldsm_x4(pa[0], pa[1], pa[2], pa[3], sP + aoff);
                ldsm_x4(sa[0], sa[1], sa[2], sa[3], sS + aoff);
#pragma unroll
                for (int d2 = 0; d2 < NH / 2; ++d2) {
                    const uint32_t boff = swz<D>(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                                 wn * (D / 16) + d2 * 2 + (lane >> 4));
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3, sO + boff);
                    mma16816(dv[2 * d2], pa, b0, b1);
                    mma16816(dv[2 * d2 + 1], pa, b2, b3);
                    ldsm_x4_t(b0, b1, b2, b3, sQ + boff);
                    mma16816(dk[2 * d2], sa, b0, b1);
                    mma16816(dk[2 * d2 + 1], sa, b2, b3);
                }
            }
            __syncthreads();  // Q and dO of this tile are no longer read

            if (qt + 1 < n_tiles) {
                load_rows<D>(sQ, a.q + (size_t)h * D, rstride,
                             [&](int r) { return tok_of(qt + 1, r); });
                load_rows<D>(sO, a.dout + (size_t)h * D, rstride,
                             [&](int r) { return tok_of(qt + 1, r); });
                cp_async_commit();
                fill_meta(qt + 1, (qt + 1) & 1);
            }

            // dQ (unscaled) += dS K: rows 16 wm .. +15 x column half wn
            float dq[NH][4];
#pragma unroll
            for (int j = 0; j < NH; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) dq[j][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kN / 16; ++ks) {
                uint32_t ra[4];
                ldsm_x4(ra[0], ra[1], ra[2], ra[3],
                        sR + swz<64>(wm * 16 + (lane & 15), ks * 2 + (lane >> 4)));
#pragma unroll
                for (int d2 = 0; d2 < NH / 2; ++d2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(b0, b1, b2, b3,
                              sK + swz<D>(ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                          wn * (D / 16) + d2 * 2 + (lane >> 4)));
                    mma16816(dq[2 * d2], ra, b0, b1);
                    mma16816(dq[2 * d2 + 1], ra, b2, b3);
                }
            }
            // lane pairs (t, t ^ 1) swap halves: the even lane adds columns
            // 2t .. 2t+3 of row g, the odd lane columns 2t-2 .. 2t+1 of row g+8
            const bool odd = t & 1;
            const int row_l = wm * 16 + g + (odd ? 8 : 0);
            const int tok = m_tok[row_l];
            float *dst = a.dq_acc + ((size_t)(tok < 0 ? 0 : tok) * H + h) * D + wn * (D / 2) +
                         2 * (t & ~1);
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                const float x = odd ? dq[nt][0] : dq[nt][2];
                const float y = odd ? dq[nt][1] : dq[nt][3];
                const float rx = __shfl_xor_sync(0xffffffffu, x, 1);
                const float ry = __shfl_xor_sync(0xffffffffu, y, 1);
                const float4 v4 = odd ? make_float4(rx, ry, dq[nt][2], dq[nt][3])
                                      : make_float4(dq[nt][0], dq[nt][1], rx, ry);
                if (tok >= 0) atomicAdd(reinterpret_cast<float4 *>(dst + nt * 8), v4);
            }
        }
        __syncthreads();  // K and dS are no longer read: the next unit may load

#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int kl = wm * 16 + g + 8 * hh;
            if (kl >= nkeys) continue;
            const size_t o = ((size_t)(key0 + kl) * H + h) * D + wn * (D / 2) + 2 * t;
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                *reinterpret_cast<__nv_bfloat162 *>(a.dk + o + nt * 8) =
                    __floats2bfloat162_rn(dk[nt][2 * hh] * a.scale, dk[nt][2 * hh + 1] * a.scale);
                *reinterpret_cast<__nv_bfloat162 *>(a.dv + o + nt * 8) =
                    __floats2bfloat162_rn(dv[nt][2 * hh], dv[nt][2 * hh + 1]);
            }
        }
    }
}

__global__ void __launch_bounds__(256) bwd_dq_kernel(const float4 *__restrict__ acc,
                                                     uint2 *__restrict__ dq, long long n4,
                                                     float scale) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 x = acc[i];
        __nv_bfloat162 lo = __floats2bfloat162_rn(x.x * scale, x.y * scale);
        __nv_bfloat162 hi = __floats2bfloat162_rn(x.z * scale, x.w * scale);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t *>(&lo);
        w.y = *reinterpret_cast<uint32_t *>(&hi);
        dq[i] = w;
    }
}

}  // namespace bwd


template <int D>
static cudaError_t launch_bwd_d(const Plan &p, const Workspace &ws, const bwd::Args &a,
                                const __nv_bfloat16 *out, cudaStream_t st) {
    using namespace bwd;
    const long long rows = (long long)p.total * p.H;
    cudaError_t e = cudaSuccess;
    if (bwd_tc_supported(p)) {
        // dk, dv and the dq accumulator on the tcgen05 tensor cores
        e = launch_bwd_kv_tc(p, ws, a.q, a.k, a.v, a.lse, a.dout, a.dk, a.dv, st);
    } else {
        constexpr int smem = smem_bytes<D>();
        cudaFuncSetAttribute(bwd_kv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        const long long grid = a.n_units < (1ll << 30) ? a.n_units : (1ll << 30);
        bwd_kv_kernel<D><<<(unsigned)grid, kThreads, smem, st>>>(a);
        note_launches(1);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const long long n4 = rows * D / 4;
    const long long blocks = (n4 + 255) / 256;
    const int cap = sm_count() * 8;
    bwd_dq_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, st>>>(
        reinterpret_cast<const float4 *>(ws.dq_acc), reinterpret_cast<uint2 *>(a.dq_out), n4,
        a.scale);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_bwd_delta(const Plan &p, const Workspace &ws, const __nv_bfloat16 *out,
                             const __nv_bfloat16 *dout, cudaStream_t st) {
    const long long rows = (long long)p.total * p.H;
    const long long warps_needed = (rows + 4 * (256 / p.D) - 1) / (4 * (256 / p.D));
    const long long blocks = std::min<long long>((warps_needed + 7) / 8, 16ll * sm_count());
    if (p.D == 64)
        bwd::bwd_delta_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(out, dout, ws.delta, rows, p.H,
                                                                    p.total);
    else
        bwd::bwd_delta_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(out, dout, ws.delta, rows,
                                                                     p.H, p.total);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                            const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                            const __nv_bfloat16 *out, const float *lse,
                            const __nv_bfloat16 *dout, __nv_bfloat16 *dq, __nv_bfloat16 *dk,
                            __nv_bfloat16 *dv, cudaStream_t st) {
    bwd::Args a;
    a.g.cu = ws.cu;
    a.g.blk_base = ws.blk_base;
    a.g.bad = ws.bad;
    a.g.num_seqs = p.num_seqs;
    a.g.total = p.total;
    a.g.H = p.H;
    a.g.D = p.D;
    a.g.bs = p.bs;
    a.q = q;
    a.k = k;
    a.v = v;
    a.dout = dout;
    a.lse = lse;
    a.delta = ws.delta;
    a.dq_acc = ws.dq_acc;
    a.dq_out = dq;
    a.dk = dk;
    a.dv = dv;
    a.fixed = p.fixed ? 1 : 0;
    a.S_fixed = p.max_len;
    a.dense = p.dense ? 1 : 0;
    a.km1 = p.km1;
    a.list = ws.list;
    a.list_off = ws.list_off;
    a.tiles_per_block = p.bs / bwd::kN;
    a.n_units = (long long)p.NBcap * p.H * a.tiles_per_block;
    a.scale = (float)(1.0 / __builtin_sqrt((double)p.D));
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)p.D));
    return p.D == 64 ? launch_bwd_d<64>(p, ws, a, out, st) : launch_bwd_d<128>(p, ws, a, out, st);
}

}  // namespace moba
