// moba_gate_tc.cu -- gate + top-k with the block scores on the tensor cores.
//
// Pages: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) sections 3.1
// and 4.1 (mean-pooled block representation, future blocks masked, top_k of
// the sorted block scores); "MOBA mixture of block attention for
// server-side long context" (hncyxsy.com/news/197418) section 3 (current
// block forced; inner product with the mean-pooled keys).
//
// Persistent: one CTA per SM walks a contiguous range of units, a unit being
// 128 consecutive query rows of one (sequence, head).  Units are ordered
// sequence, head, row tile (the tiles of a head alternate from both ends so a
// range mixes cheap early rows with costly late ones), so a CTA keeps the
// pooled keys of one head resident for many units.  Roles:
//   warp 0      TMA: a ring of q tiles (as many stages as the shared memory
//               left beside the keys holds) and, whenever the (sequence, head)
//               changes, the head's pooled keys split into two bf16 terms,
//               kbar ~= hi + lo (hi = bf16(kbar), lo = bf16(kbar - hi)); it
//               leaves each unit's fields beside its q stage;
//   warp 1      allocates TMEM; lane 0 issues one MMA chain per unit,
//               approx[r][c] = q_r . hi_c + q_r . lo_c (M128, N = the unit's
//               scored blocks rounded up to 16, fp32 in TMEM), into as many
//               TMEM slots as the longest sequence's block count allows;
//   warps 2 ..  NWG selection warpgroups taking units in turn; thread r owns
//               row r (its TMEM lane):
//     1. keeps the k largest approximate scores of its row.  With
//        |approx - exact| <= E, E = 2^-13 ||q_r|| max_c ||kbar_c|| (at least
//        8x the worst case of the bf16 split, the fp32 MMA accumulation and
//        the fp32 dot product): when the k-th is below T - 2E (T the (k-1)-th)
//        the blocks with approx >= T are the exact top k-1 and the row is
//        written here, with its selections added into the per-list counts;
//     2. otherwise the row and its candidates (approx >= T - 2E: they hold
//        the exact top k-1, and every other block scores below all of them)
//        go to gate_exact_kernel, which scores them exactly with the summation
//        order of the CUDA-core gate (four lane partials of four interleaved
//        sums), so the selection -- and its lower-index tie-break -- equals
//        that kernel's bit for bit.
// Rows whose own block has at most k-1 predecessors take them all.
// The MMA lane polls its barriers, the other roles wait suspended.  Every
// wait is bounded; a wait that runs out records MOBA_ERR_TIMEOUT.
#include <algorithm>

#include "moba.h"
#include "moba_internal.cuh"
#include "moba_ptx.cuh"
#include "moba_select.cuh"

namespace moba {
namespace gate_tc {
using namespace ptx;
using sel::exact_score;
using sel::kEmpty;
using sel::top_insert;

constexpr int kRows = 128;                     // query rows per unit (the MMA's M)
// TMA warp, MMA warp and NWG selection warpgroups (three when the top lists
// are short enough to fit the register budget of 16 warps, else two)
__host__ __device__ constexpr int threads_for(int nwg) { return 64 + 128 * nwg; }
constexpr int kMaxQ = 6;                       // q stages at most
#ifndef MOBA_GATE_NWG_SHORT
#define MOBA_GATE_NWG_SHORT 4
#endif
// selection warpgroups when the top lists hold at most two blocks
constexpr int kNwgShort = MOBA_GATE_NWG_SHORT;
constexpr int kMaxSlots = 8;                   // TMEM score slots at most
constexpr int kMaxBlocks = 256;                // blocks per sequence
// Rows left to the exact kernel carry up to 8 candidate blocks packed one byte
// each with 0xff as the empty marker: past candidates are below the own block,
// so at most kMaxBlocks - 2 = 254, and a candidate id of 255 -- which would
// read as empty -- cannot occur while the cap holds.
static_assert(kMaxBlocks <= 256, "candidate block ids are packed into one byte each");

struct Args {
    Geometry g;
    const __nv_bfloat16 *q;  // [total][H][D]
    int *counts;             // [NB * H] selections per (block, head), or nullptr
    // rows the score margin cannot settle, for the exact kernel: two words per
    // row, the row (token * H + head, bit 62 set when every past block is a
    // candidate) and up to 8 candidate blocks, one byte each, ascending (0xff
    // = none).  CTA b writes its rows from row u0_b * 128 on (u0_b its first
    // unit: room for all of its rows) and their number into need_count[b].
    unsigned long long *need_list;
    int *need_count;
    const int *gtile;    // [num_seqs + 1] 128-row tiles before each sequence
    const float *kbar;   // [NB][H][D] fp32
    const float *knorm;  // [NB][H] L2 norms of the pooled keys
    int32_t *idx;
    int topk;
    // layout chosen by the host from the longest sequence's block count W
    // (64, 128 or 256): nslots units in flight in TMEM, kb_rows = pooled-key
    // rows kept resident per term, nq q stages in the shared memory left.
    // cat (W = 64): each 64-dim box holds the 64 hi rows followed by the 64
    // lo rows, so one MMA chain with N = 128 scores q against both terms
    // (columns c and 64 + c of a slot hold q.hi_c and q.lo_c); otherwise two
    // chains accumulate q.hi and q.lo into the same columns.
    int nq, nslots, kb_rows, cat;
    int *status;
    long long wait_limit;
};

template <int D>
struct Smem {
    static constexpr int NB = D / 64;
    static constexpr uint32_t kQBox = kRows * 128;       // 128 rows x 64 dims
    static constexpr uint32_t kQStage = NB * kQBox;
    // tiles from a 1024-byte aligned base: nq q stages, then hi and lo, each
    // NB boxes of kb_rows x 64 dims
    // mbarriers: q_full[kMaxQ], q_empty[kMaxQ], kb_full, kb_empty,
    // s_full[kMaxSlots], s_empty[kMaxSlots], drain; then the TMEM address slot,
    // the abort flag, the count of rows left to the exact kernel and, per q
    // stage, the fields of the unit it holds (StageMeta, written by the
    // producer before it arms the stage's barrier)
    static constexpr int kBarQF = 0, kBarQE = kBarQF + kMaxQ, kBarKF = kBarQE + kMaxQ,
                         kBarKE = kBarKF + 1, kBarSF = kBarKE + 1, kBarSE = kBarSF + kMaxSlots,
                         kBarDrain = kBarSE + kMaxSlots, kNumBars = kBarDrain + 1;
    static constexpr uint32_t kMisc = kNumBars * 8 + 16 + 32 * kMaxQ;
    // the misc words go into the alignment slack when it is large enough, else
    // after the tiles
    static constexpr uint32_t kTileBudget = 227 * 1024 - 1008 - kMisc;
    __host__ __device__ static uint32_t kb_bytes(int kb_rows) { return 2u * NB * kb_rows * 128; }
    __host__ __device__ static uint32_t tiles(int nq, int kb_rows) {
        return nq * kQStage + kb_bytes(kb_rows);
    }
};

struct Unit {
    int b, h, t, seq0, L, bbase, nb, cmax;
};

// A unit's fields as the producer leaves them beside its q stage: the MMA lane
// and the selection warpgroups read them after the stage's barrier (no unit
// decoding, no integer division per unit or row there).
struct StageMeta {
    int cmax;       // blocks scored by some row of the unit (0: none)
    int h, t, seq0, L, bbase, nb;
    int c0;         // block of the unit's first row
};
static_assert(sizeof(StageMeta) == 32, "eight words per stage");

// unit u -> (sequence, head, row tile); cmax = blocks scored by some row of
// the tile (0 when no row is scored).  Each role walks increasing units and
// keeps the current sequence's table entries in registers, so only crossing
// into another sequence reads memory.
struct UnitCursor {
    int b = -1, nt = 0, seq0 = 0, L = 0, bbase = 0;
    int ub0 = 0, ub1 = 0;  // units of sequence b: [ub0, ub1)

    __device__ __forceinline__ void unit(const Args &a, int u, int km1, Unit &U) {
        const int H = a.g.H;
        if (b < 0 || u >= ub1) {
            int lo = 0, hi = a.g.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(a.gtile + mid) * H <= u) lo = mid; else hi = mid - 1;
            }
            b = lo;
            const int tb = __ldg(a.gtile + lo);
            nt = __ldg(a.gtile + lo + 1) - tb;
            ub0 = tb * H;
            ub1 = ub0 + nt * H;
            seq0 = __ldg(a.g.cu + lo);
            L = __ldg(a.g.cu + lo + 1) - seq0;
            bbase = __ldg(a.g.blk_base + lo);
        }
        U.b = b;
        const int rem = u - ub0;
        U.h = rem / nt;
        const int tz = rem - U.h * nt;
        U.t = (tz & 1) ? nt - 1 - (tz >> 1) : (tz >> 1);
        U.seq0 = seq0;
        U.L = L;
        U.bbase = bbase;
        U.nb = (L + a.g.bs - 1) / a.g.bs;
        const int cl = (min(L, (U.t + 1) * kRows) - 1) / a.g.bs;
        U.cmax = (km1 > 0 && cl > km1) ? cl : 0;
    }
};

// bf16 element d of row r of a K-major, 128-byte-swizzled [128][D] tile
template <int D>
__device__ __forceinline__ uint32_t q_addr(uint32_t base, int r, int d) {
    const int box = d >> 6, dd = d & 63;
    return base + box * (128 * 128) + r * 128 + ((((dd >> 3) ^ (r & 7))) << 4) + (dd & 7) * 2;
}

template <int D, int KCAP, int NWG>
__global__ void __launch_bounds__(threads_for(NWG), 1)
    gate_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_hi,
                   const __grid_constant__ CUtensorMap tmap_lo, Args a) {
    using L = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = saddr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // stride between the 64-dim boxes of pooled keys; in cat mode a box holds
    // both terms
    const uint32_t kKBox = (uint32_t)a.kb_rows * 128 * (a.cat ? 2u : 1u);
    const uint32_t misc = (base - raw >= L::kMisc) ? raw : base + L::tiles(a.nq, a.kb_rows);
    uint8_t *gmisc = smem_raw + (misc - raw);
    auto bar = [&](int i) -> uint32_t { return misc + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gmisc + L::kNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gmisc + L::kNumBars * 8 + 4);
    int *need_cnt = reinterpret_cast<int *>(gmisc + L::kNumBars * 8 + 8);
    StageMeta *stage_meta = reinterpret_cast<StageMeta *>(gmisc + L::kNumBars * 8 + 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    MOBA_RETURN_IF_BAD(a.g);
    const int H = a.g.H, km1 = a.topk - 1;
    // units fit an int (checked on the host)
    const int n_units = H * __ldg(a.gtile + a.g.num_seqs);
    const int u0 = (int)((long long)n_units * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)n_units * (blockIdx.x + 1) / gridDim.x);
    if (u0 >= u1) {
        if (tid == 0) a.need_count[blockIdx.x] = 0;
        return;
    }
    Ctl ctl{abort_flag, a.status, a.wait_limit};
    const int nq = a.nq, nslots = a.nslots;
    const int nwg = min(NWG, nslots);  // selection warpgroups in use
    const uint32_t slot_cols = 512u / nslots;
    const uint32_t sQ = base, sHi = base + nq * L::kQStage;
    const uint32_t sLo = a.cat ? sHi + (uint32_t)a.kb_rows * 128 : sHi + L::NB * kKBox;

    if (tid == 0) {
        for (int s = 0; s < kMaxQ; ++s) {
            mbar_init(bar(L::kBarQF + s), 1);
            mbar_init(bar(L::kBarQE + s), 4);  // one arrival per selection warp
        }
        mbar_init(bar(L::kBarKF), 1);
        mbar_init(bar(L::kBarKE), 1);
        for (int w = 0; w < kMaxSlots; ++w) {
            mbar_init(bar(L::kBarSF + w), 1);
            mbar_init(bar(L::kBarSE + w), 4);
        }
        mbar_init(bar(L::kBarDrain), 1);
        *abort_flag = 0;
        *need_cnt = 0;
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

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int cur = -1;  // (sequence, head) whose pooled keys are resident
            int nload = 0, i = 0;
            int s = 0, qround = 0;  // q stage of unit i and i / nq
            int qpend[kMaxQ];
            for (int s = 0; s < kMaxQ; ++s) qpend[s] = -1;
            bool go = true;
            UnitCursor cur_u;
            Unit U, NU;  // this unit and the next
            cur_u.unit(a, u0, km1, U);
            for (int u = u0; go && u < u1; ++u, ++i, U = NU) {
                if (u + 1 < u1) cur_u.unit(a, u + 1, km1, NU);
                const int pair = U.b * H + U.h;
                if (pair != cur) {
                    // the MMAs that read the previous keys have completed
                    if (nload > 0 && !wait_bar(bar(L::kBarKE), (nload - 1) & 1, ctl)) {
                        go = false;
                        break;
                    }
                    // chunks of kb_rows blocks (one in cat mode, else at most 2
                    // of 128)
                    const int rows = a.cat ? a.kb_rows : 128;
                    const int nch = (U.nb + rows - 1) / rows;
                    mbar_expect_tx(bar(L::kBarKF), 2u * L::NB * nch * rows * 128);
                    for (int x = 0; x < L::NB; ++x)
                        for (int c = 0; c < nch; ++c) {
                            const uint32_t off = x * kKBox + c * rows * 128;
                            tma_load_3d(sHi + off, &tmap_hi, bar(L::kBarKF), x * 64, U.h,
                                        U.bbase + c * 128);
                            tma_load_3d(sLo + off, &tmap_lo, bar(L::kBarKF), x * 64, U.h,
                                        U.bbase + c * 128);
                        }
                    ++nload;
                    cur = pair;
                }
                if (i >= nq && !wait_fast(bar(L::kBarQE + s), (qround - 1) & 1, ctl)) {
                    go = false;
                    break;
                }
                qpend[s] = -1;
                {  // released to the selection warps by the arrive below
                    StageMeta &m = stage_meta[s];
                    m.cmax = U.cmax;
                    m.h = U.h;
                    m.t = U.t;
                    m.seq0 = U.seq0;
                    m.L = U.L;
                    m.bbase = U.bbase;
                    m.nb = U.nb;
                    m.c0 = U.t * kRows / a.g.bs;
                }
                mbar_expect_tx(bar(L::kBarQF + s), L::kQStage);
                for (int x = 0; x < L::NB; ++x)
                    tma_load_3d(sQ + s * L::kQStage + x * L::kQBox, &tmap_q, bar(L::kBarQF + s),
                                x * 64, U.h, U.seq0 + U.t * kRows);
                qpend[s] = i;
                if (++s == nq) {
                    s = 0;
                    ++qround;
                }
            }
            if (*abort_flag) {
                // let the copies still in flight land before the CTA exits
                for (int s = 0; s < kMaxQ; ++s)
                    if (qpend[s] >= 0)
                        drain_bar(bar(L::kBarQF + s), (qpend[s] / nq) & 1, a.wait_limit);
                if (nload > 0) drain_bar(bar(L::kBarKF), (nload - 1) & 1, a.wait_limit);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            int nload = 0, i = 0;
            int s = 0, qround = 0, w = 0, wround = 0;  // q stage, TMEM slot of unit i
            bool ok = true;
            // shared-memory descriptors: the start-address field (bits 0-13, in
            // 16-byte units) is advanced by plain addition below
            const uint64_t dhi = sdesc(sHi, 16, 1024), dlo = sdesc(sLo, 16, 1024);
            const uint32_t kbox16 = kKBox >> 4;
            // the unit's (sequence, head) is decoded only when it changes; the
            // scored-block count comes with the q stage
            UnitCursor cur_u;
            Unit U;
            int left = 0;  // units of the current (sequence, head) still to come
            for (int u = u0; ok && u < u1; ++u, ++i, --left) {
                if (left == 0) {
                    cur_u.unit(a, u, km1, U);
                    left = cur_u.nt - ((u - cur_u.ub0) - U.h * cur_u.nt);
                    // the previous keys may be replaced once these MMAs complete
                    if (nload > 0) tc_commit(bar(L::kBarKE));
                    if (!wait_poll(bar(L::kBarKF), nload & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    ++nload;
                }
                if (!wait_poll(bar(L::kBarQF + s), qround & 1, ctl) ||
                    (wround > 0 && !wait_poll(bar(L::kBarSE + w), (wround - 1) & 1, ctl))) {
                    ok = false;
                    break;
                }
                const int cmax = stage_meta[s].cmax;
                tc_fence_after();
                if (cmax > 0 && a.cat) {
                    // one chain: N = 128 rows of [hi; lo]
                    const uint32_t idesc = idesc_bf16(kRows, 128, 0);
                    const uint32_t tS = tmem + w * slot_cols;
                    const uint64_t dq = sdesc(sQ + s * L::kQStage, 16, 1024);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t aoff = (uint64_t)((k / 4) * (L::kQBox >> 4) + (k % 4) * 2);
                        const uint64_t boff = (uint64_t)((k / 4) * kbox16 + (k % 4) * 2);
                        tc_mma(tS, dq + aoff, dhi + boff, idesc, k > 0);
                    }
                    tc_commit(bar(L::kBarSF + w));
                } else if (cmax > 0) {
                    const int n = min((int)slot_cols, (cmax + 15) & ~15);
                    const uint32_t idesc = idesc_bf16(kRows, n, 0);
                    const uint32_t tS = tmem + w * slot_cols;
                    const uint64_t dq = sdesc(sQ + s * L::kQStage, 16, 1024);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        // 16 dims = 32 bytes = 2 units; a 64-dim box further on
                        const uint64_t aoff = (uint64_t)((k / 4) * (L::kQBox >> 4) + (k % 4) * 2);
                        const uint64_t boff = (uint64_t)((k / 4) * kbox16 + (k % 4) * 2);
                        tc_mma(tS, dq + aoff, dhi + boff, idesc, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t aoff = (uint64_t)((k / 4) * (L::kQBox >> 4) + (k % 4) * 2);
                        const uint64_t boff = (uint64_t)((k / 4) * kbox16 + (k % 4) * 2);
                        tc_mma(tS, dq + aoff, dlo + boff, idesc, 1u);
                    }
                    tc_commit(bar(L::kBarSF + w));
                } else {
                    mbar_arrive(bar(L::kBarSF + w));  // no row of the unit is scored
                }
                if (++s == nq) {
                    s = 0;
                    ++qround;
                }
                if (++w == nslots) {
                    w = 0;
                    ++wround;
                }
            }
            // every MMA this thread issued has finished before TMEM is freed
            tc_commit(bar(L::kBarDrain));
            drain_bar(bar(L::kBarDrain), 0, a.wait_limit);
        }
        __syncwarp();
    } else {
        // ================= selection (warps 2 ..) =================
        // warpgroup wg takes units wg, wg + nwg, ...; no more warpgroups than
        // TMEM slots
        const int wg = (warp - 2) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;  // my TMEM lane and q row
        const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);
        int kn_pair = -1;  // (sequence, head) whose key-norm maximum is in kn
        float kn = 0.f;
        for (int u = u0 + wg, i = wg; wg < nwg && u < u1; u += nwg, i += nwg) {
            const int s = i % nq, slot = i % nslots;
            const uint32_t tS = tlane + slot * slot_cols;
            const uint32_t sq = sQ + s * L::kQStage;
            // the unit's fields, copied before the stage is handed back
            if (!__all_sync(0xffffffffu, wait_fast(bar(L::kBarQF + s), (i / nq) & 1, ctl))) break;
            Unit U;
            {
                const StageMeta &m = stage_meta[s];
                U.cmax = m.cmax;
                U.h = m.h;
                U.t = m.t;
                U.seq0 = m.seq0;
                U.L = m.L;
                U.bbase = m.bbase;
                U.nb = m.nb;
                U.b = m.c0;  // (the block of the unit's first row, below)
            }
            const int my_i = U.t * kRows + row;
            const bool valid = my_i < U.L;
            // my row's block: the unit's 128 rows span at most three blocks
            // (block sizes are multiples of 64)
            const int x_in = U.t * kRows - U.b * a.g.bs + row;
            const int ci = valid ? U.b + (x_in >= a.g.bs) + (x_in >= 2 * a.g.bs) : 0;
            const int tok = U.seq0 + my_i;
            const bool scored = valid && km1 > 0 && ci > km1;
            // largest pooled-key norm of the head's blocks (the margin), once per
            // (sequence, head)
            const int pair = U.bbase * H + U.h;
            if (pair != kn_pair) {
                kn = 0.f;
                for (int c = lane; c < U.nb; c += 32)
                    kn = fmaxf(kn, __ldg(a.knorm + (size_t)(U.bbase + c) * H + U.h));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) kn = fmaxf(kn, __shfl_xor_sync(0xffffffffu, kn, o));
                kn_pair = pair;
            }

            int ti[KCAP];  // selected past blocks, ascending, at the top end
#pragma unroll
            for (int x = 0; x < KCAP; ++x) ti[x] = kEmpty;
            bool need = false;  // the exact kernel writes this row
            unsigned long long cand = ~0ull;  // its candidate blocks, one byte each
            int ncand = 0;
            // ||q_r||^2 for the margin, from the q stage while the unit's MMAs
            // run: four independent f32x2 accumulators (a bf16 is the top half
            // of its fp32)
            float qq = 0.f;
            if (scored) {
                float2 acc[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int d = 0; d < D; d += 8) {
                    uint32_t w[4];
                    // volatile: kept after the wait for the stage's barrier
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(q_addr<D>(sq, row, d)));
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = make_float2(__uint_as_float(w[e] << 16),
                                                     __uint_as_float(w[e] & 0xffff0000u));
                        acc[e] = ffma2(f, f, acc[e]);
                    }
                }
                qq = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                     ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
            }
            if (!__all_sync(0xffffffffu, wait_fast(bar(L::kBarSF + slot), (i / nslots) & 1, ctl))) break;
            tc_fence_after();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarQE + s));  // the MMAs have read the q stage
            // the TMEM slot is handed back right after its last read
            bool slot_held = true;
            auto release_slot = [&]() {
                if (slot_held) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(L::kBarSE + slot));
                    slot_held = false;
                }
            };
            if (U.cmax > 0) {
                // pass 1: the k largest approximate scores of the row (values only:
                // a min/max insertion network, 2k-1 operations per block)
                float tv[KCAP + 1];
#pragma unroll
                for (int x = 0; x <= KCAP; ++x) tv[x] = -INFINITY;
                // CW scores per TMEM round trip (64 when the registers allow);
                // in cat mode a score is the sum of its hi and lo columns
                constexpr int CW = NWG >= 4 ? 32 : 64;
                uint32_t v[CW / 32][32];
                auto load_chunk = [&](int c0) {
#pragma unroll
                    for (int hh = 0; hh < CW / 32; ++hh) {
                        tc_ld32(tS + c0 + 32 * hh, v[hh]);
                        if (a.cat) {  // the lo columns, 16 at a time (register budget)
#pragma unroll
                            for (int q16 = 0; q16 < 2; ++q16) {
                                uint32_t lo[16];
                                tc_ld16(tS + 64 + c0 + 32 * hh + 16 * q16, lo);
                                tc_wait_ld();
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    v[hh][16 * q16 + e] = __float_as_uint(
                                        __uint_as_float(v[hh][16 * q16 + e]) + __uint_as_float(lo[e]));
                            }
                        }
                    }
                    tc_wait_ld();
                };
                const bool one_chunk = U.cmax <= CW;
                for (int c0 = 0; c0 < U.cmax; c0 += CW) {
                    load_chunk(c0);
                    if (one_chunk) release_slot();
#pragma unroll
                    for (int e = 0; e < CW; ++e) {
                        const float x = (c0 + e < ci) ? __uint_as_float(v[e >> 5][e & 31]) : -INFINITY;
#pragma unroll
                        for (int j = KCAP; j > 0; --j) tv[j] = fmaxf(tv[j], fminf(tv[j - 1], x));
                        tv[0] = fmaxf(tv[0], x);
                    }
                }
                float T = -INFINITY, Tk = -INFINITY;
#pragma unroll
                for (int x = 0; x <= KCAP; ++x) {
                    if (x == km1 - 1) T = tv[x];
                    if (x == km1) Tk = tv[x];
                }
                const float E = 0x1p-13f * sqrtf(qq) * kn;
                // When the k-th is below T - 2E the blocks with approx >= T are
                // the exact top k-1 (exactly k-1 of them).  Otherwise the blocks
                // with approx >= T - 2E (a superset of the exact top k-1, every
                // other block scoring below all of them) go to the exact kernel.
                need = scored && !(Tk < T - 2.f * E);
                const float cut = need ? T - 2.f * E : T;
                if (__any_sync(0xffffffffu, scored)) {
                    for (int c0 = 0; c0 < U.cmax; c0 += CW) {
                        // else pass 1's only chunk is still in registers
                        if (!one_chunk) load_chunk(c0);
                        // bit e: block c0 + e is selected / a candidate
                        unsigned long long mask = 0ull;
#pragma unroll
                        for (int e = 0; e < CW; ++e)
                            if (c0 + e < ci && __uint_as_float(v[e >> 5][e & 31]) >= cut)
                                mask |= 1ull << e;
                        if (!scored) mask = 0ull;
                        while (mask) {
                            const int c = c0 + __ffsll(mask) - 1;
                            mask &= mask - 1;
                            if (need) {
                                if (ncand < 8) cand = (cand << 8) | (unsigned long long)c;
                                ++ncand;
                            } else {
                                // ascending arrival: shift in at the top end
#pragma unroll
                                for (int x = 0; x + 1 < KCAP; ++x) ti[x] = ti[x + 1];
                                ti[KCAP - 1] = c;
                            }
                        }
                    }
                }
            }
            release_slot();  // the slot is free for the warpgroup's next unit
            // rows left to the exact kernel go to this CTA's own region of the
            // list (room for all of its rows), reserved with a shared-memory count
            const unsigned nmask = __ballot_sync(0xffffffffu, need);
            if (nmask) {
                const int leader = __ffs(nmask) - 1;
                int base = 0;
                if (lane == leader) base = atomicAdd(need_cnt, __popc(nmask));
                base = __shfl_sync(0xffffffffu, base, leader);
                if (need) {
                    const size_t slot2 =
                        2 * ((size_t)u0 * kRows + base + __popc(nmask & ((1u << lane) - 1u)));
                    const unsigned long long rowid = (unsigned long long)tok * H + U.h;
                    a.need_list[slot2] = ncand > 8 ? (rowid | (1ull << 62)) : rowid;
                    a.need_list[slot2 + 1] = cand;
                }
            }

            // selected past blocks of my row, ascending, then the own block
            if (valid && !need) {
                int npast;
                int32_t *out = a.idx + ((size_t)tok * H + U.h) * a.topk;
                if (scored) {
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
#pragma unroll
                    for (int x = 0; x < KCAP; ++x)
                        if (x < npast) out[x] = ti[x];
                } else {
                    npast = (km1 == 0) ? 0 : ci;  // every past block (ci <= km1)
                    for (int x = 0; x < npast; ++x) out[x] = x;
                }
                out[npast] = ci;
                for (int x = npast + 1; x < a.topk; ++x) out[x] = -1;
            }
            // selections per (block, head): one reduction per distinct block of
            // the warp and slot
            if (a.counts && km1 > 0) {
                const int npast = (!valid || need) ? 0 : scored ? km1 : ci;
#pragma unroll
                for (int x = 0; x < KCAP; ++x) {
                    const int c = (x < npast) ? (scored ? ti[x] : x) : -1;
                    const unsigned grp = __match_any_sync(0xffffffffu, c);
                    if (c >= 0 && lane == __ffs(grp) - 1)
                        atomicAdd(a.counts + (size_t)(U.bbase + c) * H + U.h, __popc(grp));
                }
                // unscored rows with more past blocks than KCAP slots
                for (int x = KCAP; x < npast; ++x)
                    atomicAdd(a.counts + (size_t)(U.bbase + x) * H + U.h, 1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) a.need_count[blockIdx.x] = *need_cnt;
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(512)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Rows the margin could not settle, one warp each: exact fp32 scores (the
// CUDA-core gate's summation order) of the row's candidates -- or, when it had
// more than 8, of every past block -- lane l taking candidates l, l + 32, ...
// in ascending block order; the lanes' top lists are merged with k-1 warp
// arg-max rounds (score descending, block ascending) and the row is written
// like the gate's rows.
// ---------------------------------------------------------------------------
constexpr int kExactWarps = 8;
constexpr int kExactSplit = 4;  // CTAs of the exact kernel per gate CTA

template <int D, int KCAP>
__global__ void __launch_bounds__(32 * kExactWarps)
    gate_exact_kernel(Geometry g, const __nv_bfloat16 *__restrict__ q,
                      const float *__restrict__ kbar, int32_t *__restrict__ idx, int topk,
                      int *__restrict__ counts, const unsigned long long *__restrict__ need_list,
                      const int *__restrict__ need_count, const int *__restrict__ gtile,
                      int gate_ctas) {
    MOBA_RETURN_IF_BAD(g);
    const int lane = threadIdx.x & 31;
    const int km1 = topk - 1;
    // the gate's CTA cb left need_count[cb] rows from row u0_cb * 128 of the
    // list; kExactSplit CTAs share a region, warp by warp
    const int n_units = g.H * __ldg(gtile + g.num_seqs);
    const int part = blockIdx.x % kExactSplit;
    for (int cb = blockIdx.x / kExactSplit; cb < gate_ctas; cb += gridDim.x / kExactSplit) {
    const size_t region = (size_t)((long long)n_units * cb / gate_ctas) * kRows;
    const int n = need_count[cb];
    for (int w = part * kExactWarps + (threadIdx.x >> 5); w < n; w += kExactSplit * kExactWarps) {
        const size_t e = region + w;
        const unsigned long long w0 = need_list[2 * e], cand = need_list[2 * e + 1];
        const bool all = (w0 >> 62) & 1ull;
        const long long r = (long long)(w0 & ((1ull << 62) - 1));
        const int t = (int)(r / g.H), h = (int)(r % g.H);
        const int b = upper_index(g.cu, g.num_seqs, t);
        const int ci = (t - __ldg(g.cu + b)) / g.bs;
        const int bbase = __ldg(g.blk_base + b);
        const __nv_bfloat16 *qg = q + (size_t)r * D;
        const float *kb_head = kbar + ((size_t)bbase * g.H + h) * D;
        // candidate bytes were shifted in from the low end: the oldest (lowest
        // block) sits highest
        int nc = 0;
        if (!all)
            for (int x = 0; x < 8; ++x) nc += ((cand >> (8 * x)) & 0xffull) != 0xffull;
        const int ncand = all ? ci : nc;
        float ts[KCAP];
        int ti[KCAP];
#pragma unroll
        for (int x = 0; x < KCAP; ++x) {
            ts[x] = -INFINITY;
            ti[x] = kEmpty;
        }
        for (int j = lane; j < ncand; j += 32) {
            const int c = all ? j : (int)((cand >> (8 * (nc - 1 - j))) & 0xffull);
            top_insert<KCAP>(ts, ti, km1, exact_score<D>(qg, kb_head + (size_t)c * g.H * D), c);
        }
        int sel[KCAP];
#pragma unroll
        for (int x = 0; x < KCAP; ++x) {
            sel[x] = kEmpty;
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
                sel[x] = cv;
                if (ti[0] == cv) {  // the winning lane drops its head
#pragma unroll
                    for (int y = 0; y + 1 < KCAP; ++y) {
                        ts[y] = ts[y + 1];
                        ti[y] = ti[y + 1];
                    }
                    ts[KCAP - 1] = -INFINITY;
                    ti[KCAP - 1] = kEmpty;
                }
            }
        }
#pragma unroll
        for (int pass = 0; pass < KCAP; ++pass) {
#pragma unroll
            for (int x = pass & 1; x + 1 < KCAP; x += 2) {
                const int lo = min(sel[x], sel[x + 1]), hi = max(sel[x], sel[x + 1]);
                sel[x] = lo;
                sel[x + 1] = hi;
            }
        }
        if (lane == 0) {
            int32_t *out = idx + (size_t)r * topk;
#pragma unroll
            for (int x = 0; x < KCAP; ++x)
                if (x < km1) {
                    out[x] = sel[x];
                    if (counts) atomicAdd(counts + (size_t)(bbase + sel[x]) * g.H + h, 1);
                }
            out[km1] = ci;
            for (int x = km1 + 1; x < topk; ++x) out[x] = -1;
        }
    }
    }
}

}  // namespace gate_tc

bool gate_tc_supported(const Plan &p) {
    // a warpgroup's TMEM half holds 256 block scores; the selection keeps its
    // top lists in registers
    const long long nmax = (p.max_len + p.bs - 1) / p.bs;
    // the units (head x 128-row tile) are counted in an int
    const long long units = (long long)p.H * ((long long)p.total / gate_tc::kRows + p.num_seqs + 1);
    return nmax <= gate_tc::kMaxBlocks && p.topk - 1 <= 32 && (p.D == 64 || p.D == 128) &&
           units < (1ll << 31);
}


template <int D>
static cudaError_t launch_gate_tc_d(const Plan &p, const gate_tc::Args &a, const __nv_bfloat16 *q,
                                    const __nv_bfloat16 *khi, const __nv_bfloat16 *klo,
                                    cudaStream_t st) {
    CUtensorMap mq, mh, ml;
    const int kb_box = a.cat ? a.kb_rows : 128;  // pooled-key rows per TMA box
    if (!make_tma_3d(&mq, q, p.total, p.H, D, gate_tc::kRows) ||
        !make_tma_3d(&mh, khi, p.NBcap, p.H, D, kb_box) ||
        !make_tma_3d(&ml, klo, p.NBcap, p.H, D, kb_box))
        return cudaErrorInvalidValue;
    // an upper bound of the units; CTAs beyond the real count return at once
    const long long units_max =
        (long long)p.H * (((long long)p.total + gate_tc::kRows - 1) / gate_tc::kRows + p.num_seqs);
    const int grid = (int)std::min<long long>(std::min(sm_count(), kMaxGateCtas), units_max);
    const int km1 = p.topk - 1;
    using L = gate_tc::Smem<D>;
    const int smem = (int)(L::tiles(a.nq, a.kb_rows) + 1008 + L::kMisc);
#define MOBA_GATE_TC_CASE(KC)                                                                   \
    {                                                                                           \
        constexpr int nwg = (KC) <= 2 ? gate_tc::kNwgShort : (KC) <= 8 ? 3 : 2;                          \
        auto kern = gate_tc::gate_tc_kernel<D, KC, nwg>;                                        \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             smem);                                             \
        if (e != cudaSuccess) return e;                                                         \
        kern<<<grid, gate_tc::threads_for(nwg), smem, st>>>(mq, mh, ml, a);                    \
        if ((e = cudaGetLastError()) != cudaSuccess) return e;                                  \
        gate_tc::gate_exact_kernel<D, KC><<<grid * gate_tc::kExactSplit,                        \
                                            32 * gate_tc::kExactWarps, 0, st>>>(                \
            a.g, a.q, a.kbar, a.idx, a.topk, a.counts, a.need_list, a.need_count, a.gtile,    \
            grid);                                                                              \
        return cudaGetLastError();                                                              \
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
                           const float *knorm, int32_t *idx, int *counts,
                           unsigned long long *need_list, int *need_count, cudaStream_t st) {
    gate_tc::Args a;
    a.g.cu = ws.cu;
    a.g.blk_base = ws.blk_base;
    a.g.bad = ws.bad;
    a.g.num_seqs = p.num_seqs;
    a.g.total = p.total;
    a.g.H = p.H;
    a.g.D = p.D;
    a.g.bs = p.bs;
    a.q = q;
    a.counts = counts;
    a.need_list = need_list;
    a.need_count = need_count;
    a.gtile = ws.gtile;
    a.kbar = kbar;
    a.knorm = knorm;
    a.idx = idx;
    a.topk = p.topk;
    a.status = status_word();
    a.wait_limit = p.wait_limit;
    // TMEM slot width W: the longest sequence's blocks rounded up to 64, 128
    // or 256 columns; as many q stages as the shared memory left holds
    const int nmax = (p.max_len + p.bs - 1) / p.bs;
    const int W = nmax <= 64 ? 64 : nmax <= 128 ? 128 : 256;
    a.cat = W == 64 ? 1 : 0;
    a.nslots = a.cat ? 4 : 512 / W;          // a cat slot holds 64 hi + 64 lo columns
    a.kb_rows = a.cat ? 64 : W <= 128 ? 128 : 256;
    const uint32_t budget = p.D == 64 ? gate_tc::Smem<64>::kTileBudget : gate_tc::Smem<128>::kTileBudget;
    const uint32_t kb = p.D == 64 ? gate_tc::Smem<64>::kb_bytes(a.kb_rows)
                                  : gate_tc::Smem<128>::kb_bytes(a.kb_rows);
    const uint32_t qstage = p.D == 64 ? gate_tc::Smem<64>::kQStage : gate_tc::Smem<128>::kQStage;
    a.nq = std::min<int>(gate_tc::kMaxQ, (int)((budget - kb) / qstage));
    const cudaError_t e = p.D == 64 ? launch_gate_tc_d<64>(p, a, q, khi, klo, st)
                                    : launch_gate_tc_d<128>(p, a, q, khi, klo, st);
    note_launches(2);
    return e;
}

}  // namespace moba
