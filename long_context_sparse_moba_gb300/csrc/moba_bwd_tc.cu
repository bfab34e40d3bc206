// moba_bwd_tc.cu -- backward pass of MoBA attention on the sm_103a tensor
// cores: tcgen05 MMAs with the dK / dV accumulators in tensor memory, K, V,
// Q and dO staged in shared memory by TMA (the block's own rows) or by a
// cp.async gather (the rows of later blocks that selected the block).
//
// Page: "MOBA mixture of block attention for server-side long context"
// (hncyxsy.com/news/197418) section 3 trains MoBA layers end to end; the
// selection and the attention being differentiated are those of the forward
// pass ("Moonshot MoBA paper explained", gsyq.cn/news/227272, sections 3.1,
// 4.1), with the selection held fixed (top-k passes no gradient).
//
// For row i with selected keys J_i: P_ij = exp(s_ij / sqrt(D) - lse_i),
// delta_i = dO_i . O_i, dS_ij = P_ij (dO_i . v_j - delta_i);
//   dv_j = sum_i P_ij dO_i,  dk_j = sum_i dS_ij q_i / sqrt(D),
//   dq_i = sum_j dS_ij k_j / sqrt(D).
//
// Key-major and persistent: one CTA per SM walks units of 128 keys of one
// block of one head (units of the early blocks first: their lists are the
// longest).  A unit's query rows come in tiles of 64: the block's own rows
// from the unit's first key on (causal on the diagonal; on the dense path
// every later row of the sequence), then the rows of later blocks on the
// block's regroup list.  Per tile (M = 128 keys, N = 64 rows):
//   S^T  = K Q^T        (A = K, B = Q, both K-major, fp32 in TMEM)
//   dP^T = V dO^T       (A = V, B = dO)
//   P^T = 2^(S^T log2e / sqrt(D) - lse log2e), dS^T = P^T (dP^T - delta)
//   dV  += P^T dO       (A = P^T from TMEM, B = dO MN-major)
//   dK  += dS^T Q       (A = dS^T from shared memory, B = Q MN-major)
//   dQ^T = K^T dS^T     (A = K MN-major, B = dS^T MN-major; M = 128 dims)
// and the dQ^T tile (lanes = head dims, columns = rows) is re-laid by rows in
// shared memory and added into an fp32 accumulator with 16-byte reductions.
//
// Roles (320 threads):
//   warp 0      producer: K and V of the unit (TMA), per tile Q and dO (TMA
//               for own rows, a 32-lane cp.async gather for list rows) into a
//               3-stage ring, and the tile's row metadata (token, causal
//               limit, lse, delta) into shared memory;
//   warp 1      allocates TMEM; lane 0 issues the MMAs: S^T and dP^T of tile
//               n, then dV, dK and dQ^T of tile n - 1 (which waits for that
//               tile's P^T and dS^T), so one tile's MMAs run while the other
//               tile's softmax works;
//   warps 2..9  two groups of four warps: group n % 2 takes tile n.  Thread
//               = key (its TMEM lane): P^T and dS^T of its key over the 64
//               rows, P^T packed into TMEM over S^T, dS^T into shared memory;
//               then the tile's dQ^T epilogue (thread = head dim; staged by
//               rows through the group's dS^T buffer for 16-byte reductions).
//               At the end of a unit group 0 writes dV, group 1 dK.
// TMEM (512 columns): dV [0, 128), dK [128, 256), tile buffer b at 256 + 128 b:
// S^T / P^T / dQ^T in its first 64 columns, dP^T in the next 64.  dQ^T is
// written over P^T: MMAs from one thread run in order, so the dV MMA has read
// P^T before it.
// The MMA lane polls its barriers (no late wake-up of a suspended wait); the
// other roles wait suspended.  Every mbarrier wait is bounded; a wait that
// runs out records MOBA_ERR_TIMEOUT and makes every role leave its loops.
#include <cuda.h>

#include <algorithm>

#include "moba.h"
#include "moba_internal.cuh"
#include "moba_ptx.cuh"

namespace moba {
namespace bwd_tc {
using namespace ptx;

constexpr int D = 128;            // head dimension of this kernel
constexpr int kKeys = 128;        // keys per unit (the MMA's M)
constexpr int kRowsT = 64;        // query rows per tile
constexpr int kStages = 3;        // Q / dO / metadata ring
constexpr int kThreads = 64 + 256;
constexpr int kRegLaunch = 168;   // 10 warps: 65536 / 384 registers per thread
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
    Geometry g;
    const __nv_bfloat16 *q, *k, *v, *dout;
    const float *lse;           // forward lse, natural log, forward layout
    const float *delta;         // [H][total]
    const float *list_l2, *list_dl;  // per list entry: its row's lse (log2) and delta
    float *dq_acc;              // [total][H][D], zero on entry, unscaled dS K
    __nv_bfloat16 *dk, *dv;     // [total][H][D]
    int fixed, S_fixed, dense, km1;
    const int *list, *list_off; // regroup lists of the past selections
    int tiles_per_block;        // key tiles of 128 per block
    long long n_units;          // NBcap * H * tiles_per_block
    float scale, scale_log2;
    int *status;
    long long wait_limit;
};

// shared memory plan, offsets from a 1024-byte aligned base
struct Smem {
    static constexpr uint32_t kKBox = kKeys * 128;          // 128 keys x 64 dims
    static constexpr uint32_t kRBox = kRowsT * 128;         // 64 rows x 64 dims
    static constexpr uint32_t kK = 0;                       // [box 2]
    static constexpr uint32_t kV = kK + 2 * kKBox;
    static constexpr uint32_t kQ = kV + 2 * kKBox;          // [stage][box 2]
    static constexpr uint32_t kO = kQ + kStages * 2 * kRBox;
    static constexpr uint32_t kDS = kO + kStages * 2 * kRBox;  // [buffer][128 keys][64 rows]
    static constexpr uint32_t kMeta = kDS + 2 * kKeys * 128;   // [stage] tok, lim, lse2, delta
    static constexpr uint32_t kMetaStage = 4 * kRowsT * 4;
    static constexpr uint32_t kEnd = kMeta + kStages * kMetaStage;
    // mbarriers, then the TMEM address slot and the abort flag
    static constexpr int kBarKVF = 0, kBarKVE = 1, kBarQF = 2, kBarQE = kBarQF + kStages,
                         kBarMF = kBarQE + kStages, kBarME = kBarMF + kStages,
                         kBarSF = kBarME + kStages, kBarPF = kBarSF + 2, kBarDQF = kBarPF + 2,
                         kBarDQE = kBarDQF + 2, kBarAF = kBarDQE + 2, kBarAE = kBarAF + 1,
                         kBarDrain = kBarAE + 1, kNumBars = kBarDrain + 1;
    static constexpr uint32_t kMisc = kNumBars * 8 + 8;
    static constexpr uint32_t kRequest = kEnd + 1008 + kMisc;
    static_assert(kRequest <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float x) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
}
// barrier of the `count` threads of one softmax group (ids 1, 2; 0 is the CTA's)
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// instruction descriptor of kind::f16 with either operand MN-major
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One unit: 128 keys of one block of one head and the query rows that see them.
struct Unit {
    int h, b, seq0, key0, nkeys, own_end, n_own, lbeg, lcnt, n_tiles;
};

// unit u (block-major, heads inner, key tiles innermost); false when the unit
// holds no key (a key tile past a partial block's end) or lies past the last
// block (then every later unit does too: *stop is set)
__device__ __forceinline__ bool get_unit(const Args &a, long long u, int NB, Unit &U, bool *stop) {
    const int H = a.g.H;
    const int kt = (int)(u % a.tiles_per_block);
    const long long L = u / a.tiles_per_block;
    const int gblk = (int)(L / H);
    U.h = (int)(L % H);
    if (gblk >= NB) {
        *stop = true;
        return false;
    }
    U.b = upper_index(a.g.blk_base, a.g.num_seqs, gblk);
    const int c = gblk - __ldg(a.g.blk_base + U.b);
    U.seq0 = __ldg(a.g.cu + U.b);
    const int seq_end = __ldg(a.g.cu + U.b + 1);
    const int kv0 = U.seq0 + c * a.g.bs;
    const int kv_end = min(kv0 + a.g.bs, seq_end);
    U.key0 = kv0 + kt * kKeys;
    if (U.key0 >= kv_end) return false;
    U.nkeys = min(kKeys, kv_end - U.key0);
    U.own_end = a.dense ? seq_end : kv_end;
    U.n_own = (U.own_end - U.key0 + kRowsT - 1) / kRowsT;
    U.lbeg = 0;
    U.lcnt = 0;
    if (!a.dense && a.km1 > 0) {
        const int Lid = gblk * H + U.h;
        U.lbeg = __ldg(a.list_off + Lid);
        U.lcnt = __ldg(a.list_off + Lid + 1) - U.lbeg;
    }
    U.n_tiles = U.n_own + (U.lcnt + kRowsT - 1) / kRowsT;
    return true;
}

// Walks the CTA's units in order, skipping empty ones; every role uses the
// same walk, so all agree on the tile sequence.
struct UnitWalk {
    long long u;
    int NB;
    bool stop = false;
    __device__ __forceinline__ bool next(const Args &a, Unit &U) {
        while (!stop && u < a.n_units) {
            const long long cur = u;
            u += gridDim.x;
            if (get_unit(a, cur, NB, U, &stop)) return true;
        }
        return false;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_o, Args a) {
    using L = Smem;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = saddr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t misc = (base - raw >= L::kMisc) ? raw : base + L::kEnd;
    uint8_t *gmisc = smem_raw + (misc - raw);
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.g.H;
    MOBA_RETURN_IF_BAD(a.g);
    const int NB = __ldg(a.g.blk_base + a.g.num_seqs);

    const uint32_t sK = base + L::kK, sV = base + L::kV, sQ = base + L::kQ, sO = base + L::kO,
                   sDS = base + L::kDS;
    auto bar = [&](int i) -> uint32_t { return misc + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gmisc + L::kNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gmisc + L::kNumBars * 8 + 4);
    Ctl ctl{abort_flag, a.status, a.wait_limit};
    // metadata of stage s: tok[64], lim[64], lse2[64], delta[64]
    auto meta_i = [&](int s) { return reinterpret_cast<int *>(gbase + L::kMeta + s * L::kMetaStage); };
    auto meta_f = [&](int s) {
        return reinterpret_cast<float *>(gbase + L::kMeta + s * L::kMetaStage);
    };

    if (tid == 0) {
        mbar_init(bar(L::kBarKVF), 1);
        mbar_init(bar(L::kBarKVE), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(L::kBarQF + s), 32);
            mbar_init(bar(L::kBarQE + s), 1);
            mbar_init(bar(L::kBarMF + s), 32);
            mbar_init(bar(L::kBarME + s), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::kBarSF + b), 1);
            mbar_init(bar(L::kBarPF + b), 4);
            mbar_init(bar(L::kBarDQF + b), 1);
            mbar_init(bar(L::kBarDQE + b), 4);
        }
        mbar_init(bar(L::kBarAF), 1);
        mbar_init(bar(L::kBarAE), 8);
        mbar_init(bar(L::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tDV = tmem, tDK = tmem + 128;
    auto tbuf = [&](int b) -> uint32_t { return tmem + 256 + 128u * (uint32_t)b; };

    UnitWalk walk{(long long)blockIdx.x, NB};
    Unit U;

    if (warp == 0) {
        // ================= producer =================
        // Row metadata of a tile, two rows per lane; the loads of tile t + 1
        // are issued before the copies of tile t and used one tile later.
        struct TileMeta {
            int tok[2], lim[2];
            float l2[2], dl[2];
        };
        auto fetch = [&](int t, TileMeta &m) {
            const bool own = t < U.n_own;
            const int row0 = U.key0 + t * kRowsT;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = 2 * lane + j;
                m.tok[j] = -1;
                m.lim[j] = -1;
                m.l2[j] = 0.f;
                m.dl[j] = 0.f;
                if (own) {
                    const int g = row0 + r;
                    if (g < U.own_end) {
                        m.tok[j] = g;
                        m.lim[j] = min(g - U.key0, U.nkeys - 1);
                        const size_t li = a.fixed
                                              ? ((size_t)U.b * H + U.h) * a.S_fixed + (g - U.seq0)
                                              : (size_t)U.h * a.g.total + g;
                        m.l2[j] = __ldg(a.lse + li) * kLog2e;
                        m.dl[j] = __ldg(a.delta + (size_t)U.h * a.g.total + g);
                    }
                } else {
                    const int pr = (t - U.n_own) * kRowsT + r;
                    if (pr < U.lcnt) {
                        const int pos = U.lbeg + pr;
                        m.tok[j] = __ldg(a.list + pos) >> kSlotBits;
                        m.lim[j] = U.nkeys - 1;
                        m.l2[j] = __ldg(a.list_l2 + pos);
                        m.dl[j] = __ldg(a.list_dl + pos);
                    }
                }
            }
        };
        int n = 0, ui = 0;
        bool go = true;
        int kvpend = -1;                    // unit whose K/V copy is in flight
        int qpend[kStages] = {-1, -1, -1};  // tile whose Q/dO copy is in flight per stage
        // stage tile t of the unit (metadata m), fetching tile t + 1 into nx
        auto do_tile = [&](int t, const TileMeta &m, TileMeta &nx) -> bool {
            if (t + 1 < U.n_tiles) fetch(t + 1, nx);
            const int s = n % kStages;
            if (n >= kStages) {
                const uint32_t par = (uint32_t)((n / kStages - 1) & 1);
                if (!wait_fast(bar(L::kBarQE + s), par, ctl) ||
                    !wait_fast(bar(L::kBarME + s), par, ctl))
                    return false;
            }
            const bool own = t < U.n_own;
            const int row0 = U.key0 + t * kRowsT;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = 2 * lane + j;
                meta_i(s)[r] = m.tok[j];
                meta_i(s)[kRowsT + r] = m.lim[j];
                meta_f(s)[2 * kRowsT + r] = m.l2[j];
                meta_f(s)[3 * kRowsT + r] = m.dl[j];
            }
            const uint32_t q_s = sQ + s * 2 * L::kRBox, o_s = sO + s * 2 * L::kRBox;
            if (own) {
                if (lane == 0) {
                    mbar_expect_tx(bar(L::kBarQF + s), 4 * L::kRBox);
                    for (int x = 0; x < 2; ++x) {
                        tma_load_3d(q_s + x * L::kRBox, &tmap_q, bar(L::kBarQF + s), x * 64, U.h,
                                    row0);
                        tma_load_3d(o_s + x * L::kRBox, &tmap_o, bar(L::kBarQF + s), x * 64, U.h,
                                    row0);
                    }
                } else {
                    mbar_arrive(bar(L::kBarQF + s));
                }
            } else {
                // the tile's 64 rows of Q and dO, 16 bytes per lane: an instruction
                // moves 128 bytes (one box row) of each of four rows, lane ->
                // (row it * 4 + lane / 8, chunk lane % 8), into the
                // 128-byte-swizzled layout the TMA would write
                const int ch = lane & 7;
#pragma unroll 4
                for (int it = 0; it < kRowsT / 4; ++it) {
                    const int r = it * 4 + (lane >> 3);
                    const int t0 = __shfl_sync(0xffffffffu, m.tok[0], r >> 1);
                    const int t1 = __shfl_sync(0xffffffffu, m.tok[1], r >> 1);
                    const int tok = (r & 1) ? t1 : t0;
                    const bool ok = tok >= 0;
                    const size_t src_row = ((size_t)(ok ? tok : 0) * H + U.h) * D + ch * 8;
                    const uint32_t off = (uint32_t)r * 128 + ((uint32_t)(ch ^ (r & 7)) << 4);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        cp_async16(q_s + x * L::kRBox + off, a.q + src_row + x * 64, ok);
                        cp_async16(o_s + x * L::kRBox + off, a.dout + src_row + x * 64, ok);
                    }
                }
                cp_async_arrive_noinc(bar(L::kBarQF + s));
            }
            qpend[s] = n;
            mbar_arrive(bar(L::kBarMF + s));
            ++n;
            return true;
        };
        while (go && walk.next(a, U)) {
            if (ui > 0 && !wait_fast(bar(L::kBarKVE), (ui - 1) & 1, ctl)) break;
            if (lane == 0) {
                mbar_expect_tx(bar(L::kBarKVF), 4 * L::kKBox);
                for (int x = 0; x < 2; ++x) {
                    tma_load_3d(sK + x * L::kKBox, &tmap_k, bar(L::kBarKVF), x * 64, U.h, U.key0);
                    tma_load_3d(sV + x * L::kKBox, &tmap_v, bar(L::kBarKVF), x * 64, U.h, U.key0);
                }
            }
            kvpend = ui;
            // two metadata sets in turn, so a tile's loads are in flight while
            // the previous tile is staged
            TileMeta ma, mb;
            fetch(0, ma);
            for (int t = 0; go && t < U.n_tiles; t += 2) {
                go = do_tile(t, ma, mb);
                if (go && t + 1 < U.n_tiles) go = do_tile(t + 1, mb, ma);
            }
            ++ui;
        }
        if (*abort_flag) {
            // let the copies still in flight land before the CTA exits
            cp_async_wait_all();
            if (lane == 0) {
                if (kvpend >= 0) drain_bar(bar(L::kBarKVF), kvpend & 1, a.wait_limit);
                for (int s = 0; s < kStages; ++s)
                    if (qpend[s] >= 0)
                        drain_bar(bar(L::kBarQF + s), (qpend[s] / kStages) & 1, a.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t id_sdp = idesc(kKeys, kRowsT, 0, 0);  // S^T, dP^T
            constexpr uint32_t id_acc = idesc(kKeys, D, 0, 1);       // dV, dK (B MN-major)
            constexpr uint32_t id_dq = idesc(D, kRowsT, 1, 1);       // dQ^T (A, B MN-major)
            int n = 0, ui = 0;
            bool ok = true;
            // dV, dK and dQ^T of tile m (buffer m % 2, stage m % 3); first =
            // the unit's first tile (its dV / dK start from zero, after the
            // previous unit's accumulators were read)
            auto finish = [&](int m, bool first) -> bool {
                const int bm = m & 1, sm = m % kStages;
                if (!wait_poll(bar(L::kBarPF + bm), (m / 2) & 1, ctl)) return false;
                if (first && ui > 0 && !wait_poll(bar(L::kBarAE), (ui - 1) & 1, ctl)) return false;
                fence_proxy_async();
                tc_fence_after();
                const uint32_t q_s = sQ + sm * 2 * L::kRBox, o_s = sO + sm * 2 * L::kRBox;
                const uint32_t ds = sDS + bm * kKeys * 128;
#pragma unroll
                for (int k = 0; k < kRowsT / 16; ++k) {
                    // dV += P^T dO: P^T packed in the buffer's first 32 columns
                    tc_mma_ta(tDV, tbuf(bm) + k * 8, sdesc(o_s + k * 2048, L::kRBox, 1024), id_acc,
                              (k > 0 || !first) ? 1u : 0u);
                }
#pragma unroll
                for (int k = 0; k < kRowsT / 16; ++k) {
                    // dK += dS^T Q
                    tc_mma(tDK, sdesc(ds + k * 32, 16, 1024), sdesc(q_s + k * 2048, L::kRBox, 1024),
                           id_acc, (k > 0 || !first) ? 1u : 0u);
                }
                tc_commit(bar(L::kBarQE + sm));  // Q and dO of the stage are read
#pragma unroll
                for (int k = 0; k < kKeys / 16; ++k) {
                    // dQ^T = K^T dS^T over the unit's 128 keys
                    tc_mma(tbuf(bm), sdesc(sK + k * 2048, L::kKBox, 1024),
                           sdesc(ds + k * 2048, 8192, 1024), id_dq, k > 0);
                }
                tc_commit(bar(L::kBarDQF + bm));
                return true;
            };
            while (ok && walk.next(a, U)) {
                if (!wait_poll(bar(L::kBarKVF), ui & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int t = 0; t < U.n_tiles; ++t, ++n) {
                    const int s = n % kStages, b = n & 1;
                    if (!wait_poll(bar(L::kBarQF + s), (n / kStages) & 1, ctl) ||
                        (n >= 2 && !wait_poll(bar(L::kBarDQE + b), ((n - 2) / 2) & 1, ctl))) {
                        ok = false;
                        break;
                    }
                    // gathered rows were written by cp.async (generic proxy)
                    fence_proxy_async();
                    tc_fence_after();
                    const uint32_t q_s = sQ + s * 2 * L::kRBox, o_s = sO + s * 2 * L::kRBox;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ko = (uint32_t)(k / 4) * L::kKBox + (uint32_t)(k % 4) * 32;
                        const uint32_t ro = (uint32_t)(k / 4) * L::kRBox + (uint32_t)(k % 4) * 32;
                        tc_mma(tbuf(b), sdesc(sK + ko, 16, 1024), sdesc(q_s + ro, 16, 1024), id_sdp,
                               k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ko = (uint32_t)(k / 4) * L::kKBox + (uint32_t)(k % 4) * 32;
                        const uint32_t ro = (uint32_t)(k / 4) * L::kRBox + (uint32_t)(k % 4) * 32;
                        tc_mma(tbuf(b) + 64, sdesc(sV + ko, 16, 1024), sdesc(o_s + ro, 16, 1024),
                               id_sdp, k > 0);
                    }
                    tc_commit(bar(L::kBarSF + b));
                    if (t > 0 && !finish(n - 1, t == 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                if (!finish(n - 1, U.n_tiles == 1)) {
                    ok = false;
                    break;
                }
                tc_commit(bar(L::kBarKVE));  // K and V are read once these complete
                tc_commit(bar(L::kBarAF));
                ++ui;
            }
            // every MMA this thread issued has finished before TMEM is freed
            tc_commit(bar(L::kBarDrain));
            drain_bar(bar(L::kBarDrain), 0, a.wait_limit);
        }
        __syncwarp();
    } else {
        // ================= softmax, dQ epilogue, dK / dV (warps 2..9) =================
        const int wg = (warp - 2) >> 2, quarter = warp & 3;
        const int kl = quarter * 32 + lane;  // my key (and, in the dQ epilogue, my head dim)
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tb = tbuf(wg) + lane_off;
        const uint32_t ds_row = sDS + (uint32_t)wg * kKeys * 128 + (uint32_t)kl * 128;
        int n = 0, ui = 0;
        bool ok = true;
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        while (ok && walk.next(a, U)) {
            for (int t = 0; t < U.n_tiles; ++t, ++n) {
                if ((n & 1) != wg) continue;
                const int s = n % kStages;
                const int *mtok = meta_i(s), *mlim = meta_i(s) + kRowsT;
                const float *ml2 = meta_f(s) + 2 * kRowsT, *mdl = meta_f(s) + 3 * kRowsT;
                if (!__all_sync(0xffffffffu, wait_fast(bar(L::kBarMF + s), (n / kStages) & 1, ctl)) ||
                    !__all_sync(0xffffffffu, wait_fast(bar(L::kBarSF + wg), (n / 2) & 1, ctl))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // two halves of 32 rows; each half's P^T goes over S^T columns
                // that are already read, its dS^T into four 16-byte chunks of my
                // key's row of the 128-byte-swizzled K-major tile
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t sv[32], dv[32], pk[16], dsk[16];
                    tc_ld32(tb + 32 * hh, sv);
                    tc_ld32(tb + 64 + 32 * hh, dv);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const int r = 32 * hh + c;
                        const int4 lim = *reinterpret_cast<const int4 *>(mlim + r);
                        const float4 l2 = *reinterpret_cast<const float4 *>(ml2 + r);
                        const float4 dl = *reinterpret_cast<const float4 *>(mdl + r);
                        const int lims[4] = {lim.x, lim.y, lim.z, lim.w};
                        const float dls[4] = {dl.x, dl.y, dl.z, dl.w};
                        const float2 x0 = ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                                                sc2, make_float2(-l2.x, -l2.y));
                        const float2 x1 = ffma2(make_float2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])),
                                                sc2, make_float2(-l2.z, -l2.w));
                        const float xs[4] = {x0.x, x0.y, x1.x, x1.y};
                        float p[4], dsv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            p[e] = (kl <= lims[e]) ? fast_exp2(xs[e]) : 0.f;
                            dsv[e] = p[e] * (__uint_as_float(dv[c + e]) - dls[e]);
                        }
                        __nv_bfloat162 p01 = __floats2bfloat162_rn(p[0], p[1]);
                        __nv_bfloat162 p23 = __floats2bfloat162_rn(p[2], p[3]);
                        __nv_bfloat162 d01 = __floats2bfloat162_rn(dsv[0], dsv[1]);
                        __nv_bfloat162 d23 = __floats2bfloat162_rn(dsv[2], dsv[3]);
                        pk[c / 2] = *reinterpret_cast<uint32_t *>(&p01);
                        pk[c / 2 + 1] = *reinterpret_cast<uint32_t *>(&p23);
                        dsk[c / 2] = *reinterpret_cast<uint32_t *>(&d01);
                        dsk[c / 2 + 1] = *reinterpret_cast<uint32_t *>(&d23);
                    }
                    tc_st16(tb + 16 * hh, pk);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int ch = 4 * hh + q4;
                        st_shared_v4(ds_row + ((uint32_t)(ch ^ (kl & 7)) << 4), dsk[4 * q4],
                                     dsk[4 * q4 + 1], dsk[4 * q4 + 2], dsk[4 * q4 + 3]);
                    }
                }
                tc_wait_st();
                fence_proxy_async();  // the MMAs read dS^T through the async proxy
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kBarPF + wg));

                // dQ^T of the tile, lane = head dim kl, column = row: re-laid by
                // rows through this group's dS^T buffer (free once the dQ^T MMAs
                // have completed), 32 rows at a time, then added into the fp32
                // accumulator with 16-byte reductions, a warp covering one row's
                // 128 dims per instruction
                if (!__all_sync(0xffffffffu, wait_fast(bar(L::kBarDQF + wg), (n / 2) & 1, ctl))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t q0[32], q1[32];
                tc_ld32(tb, q0);
                tc_ld32(tb + 32, q1);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kBarDQE + wg));
                // rows quarter * 8 + i of each pass are this warp's to reduce
                int rtok[2][8];
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int4 t0 = *reinterpret_cast<const int4 *>(mtok + 32 * pass + quarter * 8);
                    const int4 t1 = *reinterpret_cast<const int4 *>(mtok + 32 * pass + quarter * 8 + 4);
                    rtok[pass][0] = t0.x; rtok[pass][1] = t0.y; rtok[pass][2] = t0.z; rtok[pass][3] = t0.w;
                    rtok[pass][4] = t1.x; rtok[pass][5] = t1.y; rtok[pass][6] = t1.z; rtok[pass][7] = t1.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kBarME + s));  // the tile's metadata is read
                const uint32_t stg = sDS + (uint32_t)wg * kKeys * 128;
                float *dq_h = a.dq_acc + (size_t)U.h * D + 4 * lane;
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        st_shared_f32(stg + (uint32_t)c * 512 + (uint32_t)kl * 4,
                                      __uint_as_float(pass == 0 ? q0[c] : q1[c]));
                    named_bar_sync(1 + wg, 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int tk = rtok[pass][i];
                        const uint4 v4 = ld_shared_v4(stg + (uint32_t)(quarter * 8 + i) * 512 + lane * 16);
                        if (tk >= 0)
                            atomicAdd(reinterpret_cast<float4 *>(dq_h + (size_t)tk * H * D),
                                      make_float4(__uint_as_float(v4.x), __uint_as_float(v4.y),
                                                  __uint_as_float(v4.z), __uint_as_float(v4.w)));
                    }
                    named_bar_sync(1 + wg, 128);  // the staging rows may be written again
                }
            }
            if (!ok) break;
            // the unit's dV (group 0) and dK (group 1): thread = key
            if (!__all_sync(0xffffffffu, wait_fast(bar(L::kBarAF), ui & 1, ctl))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = (wg == 0 ? tDV : tDK) + lane_off;
            __nv_bfloat16 *dst = (wg == 0 ? a.dv : a.dk) + ((size_t)(U.key0 + kl) * H + U.h) * D;
            const float f = wg == 0 ? 1.f : a.scale;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t x[32];
                tc_ld32(tacc + c0, x);
                tc_wait_ld();
                if (kl < U.nkeys) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(x[c + 2 * e]) * f,
                                                                      __uint_as_float(x[c + 2 * e + 1]) * f);
                            w[e] = *reinterpret_cast<uint32_t *>(&bb);
                        }
                        *reinterpret_cast<uint4 *>(dst + c0 + c) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarAE));
            ++ui;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                     : "memory");
    }
}

}  // namespace bwd_tc

bool bwd_tc_supported(const Plan &p) { return p.D == bwd_tc::D && p.attn_kind == MOBA_ATTN_TCGEN05; }

cudaError_t launch_bwd_kv_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                             const float *lse, const __nv_bfloat16 *dout, __nv_bfloat16 *dk,
                             __nv_bfloat16 *dv, cudaStream_t st) {
    using namespace bwd_tc;
    CUtensorMap mk, mv, mq, mo;
    if (!make_tma_3d(&mk, k, p.total, p.H, D, kKeys) || !make_tma_3d(&mv, v, p.total, p.H, D, kKeys) ||
        !make_tma_3d(&mq, q, p.total, p.H, D, kRowsT) ||
        !make_tma_3d(&mo, dout, p.total, p.H, D, kRowsT))
        return cudaErrorInvalidValue;
    Args a;
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
    a.list_l2 = ws.list_l2;
    a.list_dl = ws.list_dl;
    a.dq_acc = ws.dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.fixed = p.fixed ? 1 : 0;
    a.S_fixed = p.max_len;
    a.dense = p.dense ? 1 : 0;
    a.km1 = p.km1;
    a.list = ws.list;
    a.list_off = ws.list_off;
    a.tiles_per_block = (p.bs + kKeys - 1) / kKeys;
    a.n_units = (long long)p.NBcap * p.H * a.tiles_per_block;
    a.scale = (float)(1.0 / __builtin_sqrt((double)D));
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    a.status = status_word();
    a.wait_limit = p.wait_limit;
    auto kern = bwd_tc_kernel;
    static int checked = 0;
    if (!checked) {
        cudaFuncAttributes fa;
        cudaError_t e0 = cudaFuncGetAttributes(&fa, kern);
        if (e0 != cudaSuccess) return e0;
        checked = (fa.numRegs <= kRegLaunch && fa.maxThreadsPerBlock >= kThreads) ? 1 : -1;
    }
    if (checked < 0) return cudaErrorInvalidConfiguration;
    const int smem = (int)Smem::kRequest;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long grid = std::min<long long>(sm_count(), a.n_units);
    kern<<<(unsigned)(grid > 0 ? grid : 1), kThreads, smem, st>>>(mk, mv, mq, mo, a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moba
