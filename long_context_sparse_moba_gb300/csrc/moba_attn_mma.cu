// moba_attn_mma.cu -- block-sparse attention on the warp-level bf16 MMA path
// (mma.sync m16n8k16, fp32 accumulate): the portable first path, kept as the
// correctness baseline next to the tcgen05 kernels.
//
// Two kernels share one tile loop (64 query rows x 64-key tiles, online
// softmax in the log2 domain):
//   past    -- one work tile = up to 64 query rows that selected the same past
//              block of the same head (gathered through the regroup lists);
//              writes a normalised partial output and its log2-sum-exp per
//              (row, slot).
//   current -- one work tile = 64 consecutive query rows; causal attention
//              over the own block (or, on the dense path, over every key up to
//              the row), then the log-sum-exp merge with the row's past
//              partials; writes bf16 out and fp32 lse.
// Pages: "When a MoBA reproduction will not run" (mhpq.cn/news/582794) section
// 3.3 (attention over the batched selected blocks, causal mask inside the
// current block) and "MOBA mixture of block attention for server-side long
// context" (hncyxsy.com/news/197418) section 3 (force_current_block).
#include "moba_internal.cuh"
#include "moba_mma.cuh"

namespace moba {

namespace mma_path {

using namespace mma;

constexpr int kM = 64;        // query rows per CTA (4 warps x 16)
constexpr int kN = 64;        // keys per tile
constexpr int kThreads = 128;

struct Args {
    Geometry g;
    const __nv_bfloat16 *q, *k, *v;
    __nv_bfloat16 *out;
    float *lse;
    int topk, km1, dense, fixed, S_fixed;
    const int32_t *idx;
    const int *list, *list_off, *tile_off;
    int n_lists;
    __nv_bfloat16 *part_o;
    float *part_lse;
    float scale_log2;
};

// Copy `rows` x D of a row-gathered bf16 matrix into a swizzled tile.
template <int D, typename RowPtr>
__device__ __forceinline__ void load_tile(uint32_t s_base, const __nv_bfloat16 *fallback,
                                          RowPtr rowptr) {
    constexpr int CH = D / 8;
#pragma unroll
    for (int j = 0; j < (kN * CH) / kThreads; ++j) {
        const int id = threadIdx.x + j * kThreads;
        const int r = id / CH, ch = id % CH;
        const __nv_bfloat16 *src = rowptr(r);
        // a masked row is zero-filled (source size 0); the address stays valid
        cp_async16(s_base + swz<D>(r, ch), src ? src + ch * 8 : fallback, src != nullptr);
    }
}

template <int D>
struct TileState {
    float o[D / 8][4];
    float m[2], l[2];
};

// The tile loop: Q (already in smem) against `ntiles` KV tiles starting at
// token `kv_tok0` of the sequence; keys past `kv_end` (exclusive, sequence
// token) or after a causal row position are masked when `causal`.
template <int D>
__device__ __forceinline__ void attend(const Args &a, int h, uint32_t sQ, uint32_t sK,
                                       uint32_t sV, int kv_tok0, int kv_end, int ntiles,
                                       bool causal, int row_pos0, TileState<D> &st) {
    constexpr int KS = D / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t rstride = (size_t)a.g.H * D;
    const __nv_bfloat16 *kh = a.k + (size_t)h * D;
    const __nv_bfloat16 *vh = a.v + (size_t)h * D;
    auto kv_rows = [&](const __nv_bfloat16 *base, int tile) {
        return [=](int r) -> const __nv_bfloat16 * {
            const int tok = kv_tok0 + tile * kN + r;
            return tok < kv_end ? base + (size_t)tok * rstride : nullptr;
        };
    };
    constexpr uint32_t kTileBytes = kN * D * 2;
    load_tile<D>(sK, kh, kv_rows(kh, 0));
    load_tile<D>(sV, vh, kv_rows(vh, 0));
    cp_async_commit();

#pragma unroll
    for (int j = 0; j < D / 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
    uint32_t qa[KS][4];
    const int row0 = warp * 16 + (lane >> 2);

    for (int kt = 0; kt < ntiles; ++kt) {
        const uint32_t buf = (kt & 1) * kTileBytes * 2;  // K and V of a stage are adjacent
        if (kt + 1 < ntiles) {
            const uint32_t nb = ((kt + 1) & 1) * kTileBytes * 2;
            load_tile<D>(sK + nb, kh, kv_rows(kh, kt + 1));
            load_tile<D>(sV + nb, vh, kv_rows(vh, kt + 1));
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
                ldsm_x4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3],
                        sQ + swz<D>(warp * 16 + (lane & 15), ks * 2 + (lane >> 4)));
        }
        const uint32_t cK = sK + buf, cV = sV + buf;
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3,
                        cK + swz<D>(np * 16 + (lane & 7) + ((lane >> 4) << 3),
                                    ks * 2 + ((lane >> 3) & 1)));
                mma16816(s[2 * np], qa[ks], b0, b1);
                mma16816(s[2 * np + 1], qa[ks], b2, b3);
            }
        }
        // scale, mask, online softmax (two rows per thread: row0, row0 + 8)
        float mx[2] = {-INFINITY, -INFINITY};
        const int key0 = kv_tok0 + kt * kN + 2 * (lane & 3);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + j * 8 + (e & 1);
                const int rp = row_pos0 + row0 + ((e >> 1) << 3);
                float x = s[j][e] * a.scale_log2;
                if (key >= kv_end || (causal && key > rp)) x = -INFINITY;
                s[j][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        float alpha[2], mu[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float mnew = fmaxf(st.m[r], mx[r]);
            mu[r] = (mnew == -INFINITY) ? 0.f : mnew;
            alpha[r] = fast_exp2(st.m[r] - mu[r]);
            st.m[r] = mnew;
            st.l[r] *= alpha[r];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = fast_exp2(s[j][e] - mu[e >> 1]);
                s[j][e] = p;
                st.l[e >> 1] += p;
            }
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            st.o[j][0] *= alpha[0];
            st.o[j][1] *= alpha[0];
            st.o[j][2] *= alpha[1];
            st.o[j][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
            uint32_t pa[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]),
                              pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                              pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                              pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3,
                          cV + swz<D>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                      dp * 2 + (lane >> 4)));
                mma16816(st.o[2 * dp], pa, b0, b1);
                mma16816(st.o[2 * dp + 1], pa, b2, b3);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
        st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
    }
}

template <int D>
__global__ __launch_bounds__(kThreads, 2) void past_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + kM * D * 2;
    const uint32_t sV = sK + kN * D * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    MOBA_RETURN_IF_BAD(a.g);
    const int total_tiles = __ldg(a.tile_off + a.n_lists);
    const int H = a.g.H;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        // list that owns this tile: largest L with tile_off[L] <= tile
        int lo = 0, hi = a.n_lists - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(a.tile_off + mid) <= tile) lo = mid; else hi = mid - 1;
        }
        const int L = lo;
        const int gblk = L / H, h = L % H;
        const int b = upper_index(a.g.blk_base, a.g.num_seqs, gblk);
        const int c = gblk - __ldg(a.g.blk_base + b);
        const int seq0 = __ldg(a.g.cu + b), seq_end = __ldg(a.g.cu + b + 1);
        const int kv0 = seq0 + c * a.g.bs;
        const int kv_end = min(kv0 + a.g.bs, seq_end);
        const int lbeg = __ldg(a.list_off + L), lcnt = __ldg(a.list_off + L + 1) - lbeg;
        const int r0 = (tile - __ldg(a.tile_off + L)) * kM;
        const int nrows = min(kM, lcnt - r0);
        const int *ent = a.list + lbeg + r0;
        load_tile<D>(sQ, a.q, [&](int r) -> const __nv_bfloat16 * {
            return r < nrows ? a.q + ((size_t)(__ldg(ent + r) >> kSlotBits) * H + h) * D : nullptr;
        });
        TileState<D> st;
        attend<D>(a, h, sQ, sK, sV, kv0, kv_end, (kv_end - kv0 + kN - 1) / kN, false, 0, st);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = warp * 16 + (lane >> 2) + r * 8;
            if (row >= nrows) continue;
            const int e = __ldg(ent + row);
            // head-major partials, [head][token][slot]
            const size_t slot = ((size_t)h * a.g.total + (e >> kSlotBits)) * a.km1 + (e & ((1 << kSlotBits) - 1));
            const float inv = 1.f / st.l[r];
            __nv_bfloat16 *dst = a.part_o + slot * D + 2 * (lane & 3);
#pragma unroll
            for (int j = 0; j < D / 8; ++j)
                *reinterpret_cast<__nv_bfloat162 *>(dst + j * 8) =
                    __floats2bfloat162_rn(st.o[j][2 * r] * inv, st.o[j][2 * r + 1] * inv);
            if ((lane & 3) == 0) a.part_lse[slot] = st.m[r] + __log2f(st.l[r]);
        }
        __syncthreads();
    }
}

template <int D>
__global__ __launch_bounds__(kThreads, 2) void current_kernel(Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + kM * D * 2;
    const uint32_t sV = sK + kN * D * 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.y, b = blockIdx.z;
    const int H = a.g.H;
    MOBA_RETURN_IF_BAD(a.g);
    const int seq0 = __ldg(a.g.cu + b), len = __ldg(a.g.cu + b + 1) - seq0;
    const int r0 = blockIdx.x * kM;
    if (r0 >= len) return;
    load_tile<D>(sQ, a.q, [&](int r) -> const __nv_bfloat16 * {
        return r0 + r < len ? a.q + ((size_t)(seq0 + r0 + r) * H + h) * D : nullptr;
    });
    const int kv_lo = a.dense ? 0 : (r0 / a.g.bs) * a.g.bs;
    const int kv_hi = min(r0 + kM, len);
    TileState<D> st;
    attend<D>(a, h, sQ, sK, sV, seq0 + kv_lo, seq0 + kv_hi, (kv_hi - kv_lo + kN - 1) / kN, true,
              seq0 + r0, st);
    const float ln2 = 0.69314718055994530942f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = warp * 16 + (lane >> 2) + r * 8;
        const int i = r0 + row;
        if (i >= len) continue;
        const int tok = seq0 + i;
        const float inv = 1.f / st.l[r];
        const float lse_cur = st.m[r] + __log2f(st.l[r]);
        float acc[D / 8][2];
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            acc[j][0] = st.o[j][2 * r] * inv;
            acc[j][1] = st.o[j][2 * r + 1] * inv;
        }
        float lse_out = lse_cur;
        if (!a.dense && a.km1 > 0) {
            const int ci = i / a.g.bs;
            const int32_t *sel = a.idx + ((size_t)tok * H + h) * a.topk;
            int np = 0;
            float mmax = lse_cur;
            for (; np < a.km1; ++np) {
                const int c = __ldg(sel + np);
                if (c < 0 || c >= ci) break;
                mmax = fmaxf(mmax, __ldg(a.part_lse + ((size_t)h * a.g.total + tok) * a.km1 + np));
            }
            if (np > 0) {
                float wsum = fast_exp2(lse_cur - mmax);
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    acc[j][0] *= wsum;
                    acc[j][1] *= wsum;
                }
                for (int s = 0; s < np; ++s) {
                    const size_t slot = ((size_t)h * a.g.total + tok) * a.km1 + s;
                    const float w = fast_exp2(__ldg(a.part_lse + slot) - mmax);
                    wsum += w;
                    const __nv_bfloat16 *src = a.part_o + slot * D + 2 * (lane & 3);
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        const float2 f = __bfloat1622float2(
                            __ldg(reinterpret_cast<const __nv_bfloat162 *>(src + j * 8)));
                        acc[j][0] = fmaf(w, f.x, acc[j][0]);
                        acc[j][1] = fmaf(w, f.y, acc[j][1]);
                    }
                }
                const float iw = 1.f / wsum;
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    acc[j][0] *= iw;
                    acc[j][1] *= iw;
                }
                lse_out = mmax + __log2f(wsum);
            }
        }
        __nv_bfloat16 *dst = a.out + ((size_t)tok * H + h) * D + 2 * (lane & 3);
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
            *reinterpret_cast<__nv_bfloat162 *>(dst + j * 8) =
                __floats2bfloat162_rn(acc[j][0], acc[j][1]);
        if ((lane & 3) == 0) {
            const size_t li = a.fixed ? ((size_t)b * H + h) * a.S_fixed + i
                                      : (size_t)h * a.g.total + tok;
            a.lse[li] = lse_out * ln2;
        }
    }
}

}  // namespace mma_path

int mma_tile_rows() { return mma_path::kM; }


static mma_path::Args make_args(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                __nv_bfloat16 *out, float *lse) {
    mma_path::Args a;
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
    a.out = out;
    a.lse = lse;
    a.topk = p.topk;
    a.km1 = p.km1;
    a.dense = p.dense ? 1 : 0;
    a.fixed = p.fixed ? 1 : 0;
    a.S_fixed = p.max_len;
    a.idx = ws.idx;
    a.list = ws.list;
    a.list_off = ws.list_off;
    a.tile_off = ws.tile_off;
    a.n_lists = p.NBcap * p.H;
    a.part_o = ws.part_o;
    a.part_lse = ws.part_lse;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)p.D));
    return a;
}

template <int D>
static cudaError_t launch_past_d(const mma_path::Args &a, cudaStream_t st) {
    using namespace mma_path;
    const int smem = (kM + 4 * kN) * D * 2;
    cudaFuncSetAttribute(past_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    past_kernel<D><<<sm_count() * 2, kThreads, smem, st>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_current_d(const Plan &p, const mma_path::Args &a, cudaStream_t st) {
    using namespace mma_path;
    const int smem = (kM + 4 * kN) * D * 2;
    cudaFuncSetAttribute(current_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    dim3 grid((p.max_len + kM - 1) / kM, p.H, p.num_seqs);
    current_kernel<D><<<grid, kThreads, smem, st>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attn_past_mma(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st) {
    if (p.dense || p.km1 == 0) return cudaSuccess;
    auto a = make_args(p, ws, q, k, v, nullptr, nullptr);
    return p.D == 64 ? launch_past_d<64>(a, st) : launch_past_d<128>(a, st);
}

cudaError_t launch_attn_current_mma(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                __nv_bfloat16 *out, float *lse, cudaStream_t st) {
    auto a = make_args(p, ws, q, k, v, out, lse);
    return p.D == 64 ? launch_current_d<64>(p, a, st) : launch_current_d<128>(p, a, st);
}

}  // namespace moba
