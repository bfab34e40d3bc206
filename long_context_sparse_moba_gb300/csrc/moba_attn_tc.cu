// moba_attn_tc.cu -- block-sparse attention on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory, K/V staged by TMA).
//
// Pages: "When a MoBA reproduction will not run" (mhpq.cn/news/582794) section
// 3.3 (softmax attention over the batched selected blocks, causal mask inside
// the current block) and "MOBA mixture of block attention for server-side long
// context" (hncyxsy.com/news/197418) section 3 (force_current_block).
//
// Persistent: one CTA per SM walks jobs blockIdx.x, + gridDim.x, ...; a job is
// up to 256 query rows held as two 128-row tiles (g = 0, 1) that share every
// 128-key K/V tile.  320 threads in four roles:
//   warp 0      TMA producers: lane 0 loads the Q tiles (own-block mode) and a
//               2-stage ring of K tiles, lane 1 a 2-stage ring of V tiles (one
//               TMA stream per thread tops out well below what the tensor core
//               consumes); the rings run ahead into the next job.  In the past
//               mode lane 0 also leaves each next job's descriptor in one of two
//               shared-memory slots for the softmax warps (a descriptor is a chain
//               of dependent table loads, which the producer, running ahead,
//               takes off their job boundary);
//   warp 1      allocates all 512 TMEM columns; lane 0 issues the MMAs
//                 S_g = Q_g K_j^T   (M128 N128 K=D, A and B from shared memory)
//                 O_g += P_g V_j    (M128 N=D K128, A = P_g from TMEM)
//               in the order PV_0(j-1), S_0(j), PV_1(j-1), S_1(j): the
//               tensor core runs one tile's MMAs while the other tile's
//               softmax works, and because MMAs from one thread execute in
//               order, S_g(j) may overwrite the TMEM columns that P_g(j-1)
//               occupies;
//   warps 2..9  softmax of tile 0 (warps 2..5) and tile 1 (6..9): thread r owns
//               row r (its TMEM lane).  Per 64-key half of S it reads the half
//               once, takes its max, raises the offset (to a whole number) only
//               when the max exceeds it by more than 8 (then O, the running sum
//               and, for the second half, the first half's P are rescaled by an
//               exact power of two), and writes P = 2^(s * scale - offset) as
//               bf16 pairs over the first 64 columns of S; the arithmetic runs
//               on packed fp32 pairs.  Epilogue per tile, rows re-laid through
//               4 KB of shared memory per warp for full-line global access.
// TMEM: S_g at columns 256g .. 256g+127 (P_g in the first 64), O_g at
// 256g+128 .. 256g+128+D.  One CTA per SM (192 KB of tiles + 32 KB of staging).
//
// Modes:
//   kPast     gathered rows: up to 256 rows of one regroup list (rows that
//             selected the same past block of the same head), jobs looked up in
//             the table the regroup scan writes; the softmax warps gather the
//             next job's Q rows with cp.async as soon as the MMA has released
//             Q_g, arriving on its barrier asynchronously; output = normalised
//             bf16 partial O and its log2-sum-exp per (row, slot);
//   kCurrent  rows [r0, r0 + 256) of a sequence: causal attention over the own
//             block (every key up to the row on the dense path), then the
//             log-sum-exp merge with the row's past partials -> bf16 out, lse.
//             Each tile only visits the K/V tiles its rows can see.
//
// The MMA lane polls its barriers (a suspended wait wakes up late, and every
// cycle it sleeps past a phase leaves the tensor core idle); the other roles
// wait suspended, leaving their issue slots to the softmax warps beside them.
// Every mbarrier wait is bounded (clock64 budget); a wait that runs out sets
// MOBA_ERR_TIMEOUT in the device status word and an abort flag that makes the
// other roles leave their loops; the producer then waits (bounded) for its
// copies in flight and the MMA lane for its MMAs before TMEM is freed.
#include <cuda.h>

#include "moba.h"
#include "moba_internal.cuh"
#include "moba_ptx.cuh"

namespace moba {
namespace tc {
using namespace ptx;

constexpr int kM = 128;           // rows per Q tile (the MMA's M)
constexpr int kG = 2;             // Q tiles (softmax groups) per CTA
constexpr int kRows = kM * kG;    // rows per job
constexpr int kN = 128;           // keys per K/V tile
constexpr int kStages = 2;        // depth of the K ring and of the V ring
constexpr int kThreads = 64 + 128 * kG;  // producers, MMA, 2 x 4 softmax warps
// Warps are budgeted four at a time, so 10 warps get 65536 / 384 registers
// each: the kernel is built for (and the host checks) 168.
constexpr int kRegLaunch = 168;
constexpr int kTmemCols = 512;
constexpr uint32_t kBox = 64;     // dims per TMA box (128 bytes of bf16)

enum Mode { kPast = 0, kCurrent = 1 };

// The softmax warps' waits at a job boundary (the job's last PV, the next
// job's first S): in the past mode, whose jobs are a few tiles long, they poll
// -- every warp of the CTA is waiting on the same chain then, and a late
// wake-up adds to it; elsewhere they wait suspended.
template <int MODE>
__device__ __forceinline__ bool boundary_wait(uint32_t bar, uint32_t parity, const Ctl &c) {
    return MODE == kPast ? wait_poll(bar, parity, c) : wait_bar(bar, parity, c);
}


struct Args {
    Geometry g;
    const __nv_bfloat16 *q;
    __nv_bfloat16 *out;
    float *lse;
    int topk, km1, dense, fixed, S_fixed;
    const int32_t *idx;
    const int *list, *list_off, *tile_off, *job_list;
    int n_lists;
    int n_jobs, n_rtiles;   // own-block mode: jobs = n_rtiles x num_seqs x H
    __nv_bfloat16 *part_o;  // partial outputs, bf16
    float *part_lse;
    float scale_log2;
    // own-block mode: fused jobs (query-major over their rows' past blocks)
    int fused;                    // job tables below are valid
    const int *job_nu, *job_ub;   // [jobs], [jobs][kMaxUnion]
    // set by the fusion test when some job is fused: of the two own-block
    // variants launched, only the one that matches runs
    const int *any_fused;
    int *status;
    long long wait_limit;  // clock64 budget of one wait
    int debug_flags;       // bit 0: the producer skips its first K/V load
};

// ----------------------------------------------------------------------------
// shared memory plan (offsets from a 1024-byte aligned base)
// ----------------------------------------------------------------------------
template <int D>
struct Smem {
    static constexpr int NB = D / kBox;                       // 64-dim boxes per row
    static constexpr uint32_t kQBox = kM * 128;               // 16 KB
    static constexpr uint32_t kKVBox = kN * 128;              // 16 KB
    static constexpr uint32_t kQ = 0;                         // [g][box]
    static constexpr uint32_t kK = kQ + kG * NB * kQBox;      // [stage][box]
    static constexpr uint32_t kV = kK + kStages * NB * kKVBox;
    static constexpr uint32_t kTiles = kV + kStages * NB * kKVBox;  // end of the tiles
    // 4 KB per softmax warp where its 32 rows are re-laid so that global
    // reads and writes of whole rows go out as full 128-byte lines
    static constexpr uint32_t kStageWarp = 4096;
    static constexpr uint32_t kStage = kTiles;
    static constexpr uint32_t kEnd = kStage + 4 * kG * kStageWarp;
    // mbarriers: q_full[g], q_empty[g], k_full[2], k_empty[2], v_full[2],
    // v_empty[2], s_full[g], p_full[g], pv_done[g], drain; then the TMEM
    // address slot and the abort flag
    static constexpr int kBarQ = 0, kBarQE = kBarQ + kG, kBarKF = kBarQE + kG,
                         kBarKE = kBarKF + kStages,
                         kBarVF = kBarKE + kStages, kBarVE = kBarVF + kStages,
                         kBarS = kBarVE + kStages, kBarP = kBarS + kG, kBarPV = kBarP + kG,
                         kBarDrain = kBarPV + kG, kBarDF = kBarDrain + 1, kBarDE = kBarDF + 2,
                         kNumBars = kBarDE + 2;
    // past mode: two slots of the next job's descriptor, written by the K
    // producer (desc_full / desc_empty above) for the softmax warps
    static constexpr uint32_t kDesc = (kNumBars * 8 + 8 + 15) & ~15u;
    static constexpr uint32_t kDescSlot = 80;  // a Job and its number
    static constexpr uint32_t kMisc = kDesc + 2 * kDescSlot;
    // The tiles need a 1024-byte aligned base; the dynamic window is at least
    // 16-byte aligned, so up to 1008 bytes of slack; the misc words go into
    // the slack when it is large enough, else right after the staging.  The
    // request keeps a single CTA per SM (it owns all of TMEM).
    static constexpr uint32_t kNeed = kEnd + 1008 + kMisc;
    static_assert(kNeed <= 227 * 1024, "shared memory per CTA");
    static constexpr uint32_t kRequest = kNeed > 120 * 1024 ? kNeed : 120 * 1024;
};

// One unit of work: up to 256 query rows and the K/V tiles they visit.
// rows: tile g holds job rows [g*128, g*128 + 128) (valid below nrows); K/V
// tiles [0, nkv) start at token kv_tok0; tile g visits K/V tiles [tb[g], te[g]).
// Fused own-block jobs visit their union blocks' tiles first (nut of them,
// bs / 128 per block), then their own tiles.
struct Job {
    int h, b, seq0, L_len, r0, nrows, kv_tok0, kv_end, kv_lo, nkv, lbeg;
    int nu;               // own-block mode: past blocks of a fused job (0: not fused)
    int tb[kG], te[kG];
};
static_assert(sizeof(Job) + 4 <= Smem<128>::kDescSlot, "a descriptor slot holds a Job and its number");

template <int MODE, bool FUSE = false>
__device__ __forceinline__ bool get_job(const Args &a, int job, Job &J) {
    const int H = a.g.H;
    if (MODE == kPast) {
        const int Lid = __ldg(a.job_list + job);
        const int gblk = Lid / H;
        J.h = Lid % H;
        J.b = upper_index(a.g.blk_base, a.g.num_seqs, gblk);
        const int c = gblk - __ldg(a.g.blk_base + J.b);
        J.seq0 = __ldg(a.g.cu + J.b);
        J.L_len = __ldg(a.g.cu + J.b + 1) - J.seq0;
        J.kv_lo = 0;
        J.kv_tok0 = J.seq0 + c * a.g.bs;
        J.kv_end = min(J.kv_tok0 + a.g.bs, J.seq0 + J.L_len);
        const int lbeg = __ldg(a.list_off + Lid);
        const int lcnt = __ldg(a.list_off + Lid + 1) - lbeg;
        J.r0 = (job - __ldg(a.tile_off + Lid)) * kRows;
        J.nrows = min(kRows, lcnt - J.r0);
        J.lbeg = lbeg + J.r0;
        J.nkv = (J.kv_end - J.kv_tok0 + kN - 1) / kN;
        J.nu = 0;
#pragma unroll
        for (int g = 0; g < kG; ++g) {
            J.tb[g] = 0;
            J.te[g] = (J.nrows > g * kM) ? J.nkv : 0;
        }
        return true;
    }
    // own-block mode: heavy (late) row tiles first
    J.h = job % H;
    const int t = job / H;
    J.b = t % a.g.num_seqs;
    const int x = a.n_rtiles - 1 - t / a.g.num_seqs;
    J.seq0 = __ldg(a.g.cu + J.b);
    J.L_len = __ldg(a.g.cu + J.b + 1) - J.seq0;
    J.r0 = x * kRows;
    if (J.r0 >= J.L_len) return false;
    J.nrows = min(kRows, J.L_len - J.r0);
    const int bs = a.g.bs;
    J.kv_lo = a.dense ? 0 : (J.r0 / bs) * bs;
    J.kv_tok0 = J.seq0 + J.kv_lo;
    J.kv_end = J.seq0 + J.r0 + J.nrows;
    J.nkv = (J.kv_end - J.kv_tok0 + kN - 1) / kN;
    J.lbeg = 0;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int first = J.r0 + g * kM, last = min(J.r0 + (g + 1) * kM, J.r0 + J.nrows) - 1;
        if (last < first) {
            J.tb[g] = J.te[g] = 0;
            continue;
        }
        const int lo_key = a.dense ? 0 : (first / bs) * bs;
        J.tb[g] = (lo_key - J.kv_lo) / kN;
        J.te[g] = (last - J.kv_lo) / kN + 1;
    }
    // a fused job's past blocks; their tiles are added by add_union_tiles when
    // the job starts (the load is in flight until then)
    J.nu = FUSE ? __ldg(a.job_nu + job) : 0;
    return true;
}

// A fused job (block size a multiple of 256: its rows share one block, so
// every one of its tiles starts at the block's first key) visits its union
// blocks' tiles before its own.
template <bool FUSE>
__device__ __forceinline__ void add_union_tiles(const Args &a, Job &J) {
    if (!FUSE || J.nu == 0) return;
    const int nut = J.nu * (a.g.bs / kN);
    J.nkv += nut;
#pragma unroll
    for (int g = 0; g < kG; ++g)
        if (J.te[g] > J.tb[g]) J.te[g] += nut;
}

// first token of K/V tile j of job J (number `job`)
template <bool FUSE>
__device__ __forceinline__ int tile_tok(const Args &a, const Job &J, int job, int j) {
    if (!FUSE) return J.kv_tok0 + j * kN;
    const int tpb = a.g.bs / kN;  // K/V tiles per block
    const int nut = J.nu * tpb;
    if (j < nut) {
        const int u = j / tpb;
        return J.seq0 + __ldg(a.job_ub + job * kMaxUnion + u) * a.g.bs + (j - u * tpb) * kN;
    }
    return J.kv_tok0 + (j - nut) * kN;
}

// Persistent kernel: one CTA per SM walks the jobs blockIdx.x, +gridDim.x,
// ...; every barrier phase is counted across jobs, the K/V rings run ahead
// into the next job, and in the past-block mode the next job's Q rows are
// gathered while the current job's partial outputs are written.
template <int D, int MODE, bool FUSE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, Args a) {
    using L = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = saddr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t misc = (base - raw >= L::kMisc) ? raw : base + L::kEnd;
    uint8_t *gmisc = smem_raw + (misc - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.g.H;
    MOBA_RETURN_IF_BAD(a.g);
    if (MODE == kCurrent && a.fused && (*a.any_fused != 0) != FUSE) return;
    const int njobs = (MODE == kPast) ? __ldg(a.tile_off + a.n_lists) : a.n_jobs;
    if ((int)blockIdx.x >= njobs) return;

    // ---------------- set-up (once per CTA) ----------------
    const uint32_t sQ = base + L::kQ, sK = base + L::kK, sV = base + L::kV;
    auto bar = [&](int i) -> uint32_t { return misc + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gmisc + L::kNumBars * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gmisc + L::kNumBars * 8 + 4);
    Ctl ctl{abort_flag, a.status, a.wait_limit};

    if (tid == 0) {
        for (int g = 0; g < kG; ++g) {
            // past mode: one asynchronous arrival per gathering thread
            mbar_init(bar(L::kBarQ + g), MODE == kPast ? kM : 1);
            mbar_init(bar(L::kBarQE + g), 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(L::kBarKF + s), 1);
            mbar_init(bar(L::kBarKE + s), 1);
            mbar_init(bar(L::kBarVF + s), 1);
            mbar_init(bar(L::kBarVE + s), 1);
        }
        for (int g = 0; g < kG; ++g) {
            mbar_init(bar(L::kBarS + g), 1);
            mbar_init(bar(L::kBarP + g), 4);
            mbar_init(bar(L::kBarPV + g), 1);
        }
        mbar_init(bar(L::kBarDrain), 1);
        for (int d = 0; d < 2; ++d) {
            mbar_init(bar(L::kBarDF + d), 1);
            mbar_init(bar(L::kBarDE + d), 4 * kG + 1);  // each softmax warp and the MMA lane
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================= TMA producers (lane 0: Q and K, lane 1: V) =================
        if (lane < 2) {
            const bool is_k = lane == 0;
            constexpr uint32_t kTileBytes = L::NB * L::kKVBox;
            const int bfull = is_k ? L::kBarKF : L::kBarVF, bempty = is_k ? L::kBarKE : L::kBarVE;
            const uint32_t ring = is_k ? sK : sV;
            const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
            int pend[kStages];  // tile (global count) whose copy is in flight per slot
            for (int s = 0; s < kStages; ++s) pend[s] = -1;
            int qpend[kG] = {-1, -1};  // own-block mode: Q phase in flight per tile
            int t = 0, qj = 0;  // K/V tiles and Q tiles loaded so far
            int dn = 0;         // past mode: descriptors handed to the softmax warps
            bool go = true;
            int job = blockIdx.x;
            Job J;
            while (job < njobs && !get_job<MODE, FUSE>(a, job, J)) job += gridDim.x;
            while (go && job < njobs) {
                add_union_tiles<FUSE>(a, J);
                // the next job's descriptor is fetched one job ahead
                int njob = job + gridDim.x;
                Job NJ;
                while (njob < njobs && !get_job<MODE, FUSE>(a, njob, NJ)) njob += gridDim.x;
                if (MODE == kPast && is_k) {
                    // and handed to the softmax warps, which would otherwise wait
                    // on the same chain of table loads at their job boundary
                    const int d = dn & 1;
                    if (dn >= 2 && !wait_bar(bar(L::kBarDE + d), ((dn - 2) >> 1) & 1, ctl)) {
                        go = false;
                        break;
                    }
                    uint8_t *slot = gmisc + L::kDesc + d * L::kDescSlot;
                    *reinterpret_cast<Job *>(slot) = NJ;
                    *reinterpret_cast<int *>(slot + sizeof(Job)) = njob;
                    mbar_arrive(bar(L::kBarDF + d));
                    ++dn;
                }
                if (MODE == kCurrent && is_k) {
                    for (int g = 0; g < kG && go; ++g) {
                        // the previous job's S_g MMAs have read Q_g before it is replaced
                        if (qj > 0 && !wait_bar(bar(L::kBarQE + g), (qj - 1) & 1, ctl)) {
                            go = false;
                            break;
                        }
                        mbar_expect_tx(bar(L::kBarQ + g), L::NB * L::kQBox);
                        for (int x = 0; x < L::NB; ++x)
                            tma_load_3d(sQ + (g * L::NB + x) * L::kQBox, &tmap_q, bar(L::kBarQ + g),
                                        x * kBox, J.h, J.seq0 + J.r0 + g * kM);
                        qpend[g] = qj;
                    }
                    if (!go) break;
                    ++qj;
                }
                for (int j = 0; j < J.nkv; ++j, ++t) {
                    const int s = t % kStages, use = t / kStages;
                    if (t >= kStages && !wait_bar(bar(bempty + s), (use - 1) & 1, ctl)) {
                        go = false;
                        break;
                    }
                    pend[s] = -1;
                    if (is_k && (a.debug_flags & 1) && t == 0) continue;  // fault-injection knob
                    mbar_expect_tx(bar(bfull + s), kTileBytes);
                    for (int x = 0; x < L::NB; ++x)
                        tma_load_3d(ring + (s * L::NB + x) * L::kKVBox, map, bar(bfull + s),
                                    x * kBox, J.h, tile_tok<FUSE>(a, J, job, j));
                    pend[s] = t;
                }
                job = njob;
                J = NJ;
            }
            if (*abort_flag) {
                // let the copies still in flight land before the CTA exits
                for (int s = 0; s < kStages; ++s)
                    if (pend[s] >= 0)
                        drain_bar(bar(bfull + s), (pend[s] / kStages) & 1, a.wait_limit);
                for (int g = 0; g < kG; ++g)
                    if (qpend[g] >= 0) drain_bar(bar(L::kBarQ + g), qpend[g] & 1, a.wait_limit);
            }
        }
        __syncwarp();  // reconverge before the CTA barrier (bar.sync is per warp)
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(kM, kN, 0);
            constexpr uint32_t idesc_o = idesc_bf16(kM, D, 1);
            int t = 0, qj = 0;          // K/V tiles consumed, jobs started
            int gt[kG] = {0, 0};        // per tile g: S/P tiles so far
            int dn = 0;                 // past mode: descriptors taken from the producer
            bool ok = true;
            int job = blockIdx.x;
            Job J;
            while (job < njobs && !get_job<MODE, FUSE>(a, job, J)) job += gridDim.x;
            while (ok && job < njobs) {
                add_union_tiles<FUSE>(a, J);
                // next descriptor, one job ahead (past mode: from the producer's slot)
                int njob = job + gridDim.x;
                Job NJ;
                if (MODE == kPast) {
                    if (!wait_poll(bar(L::kBarDF + (dn & 1)), (dn >> 1) & 1, ctl)) break;
                    const uint8_t *slot = gmisc + L::kDesc + (dn & 1) * L::kDescSlot;
                    NJ = *reinterpret_cast<const Job *>(slot);
                    njob = *reinterpret_cast<const int *>(slot + sizeof(Job));
                    mbar_arrive(bar(L::kBarDE + (dn & 1)));
                    ++dn;
                } else {
                    while (njob < njobs && !get_job<MODE, FUSE>(a, njob, NJ)) njob += gridDim.x;
                }
                // a Q tile without S MMAs in this job is released at once
#pragma unroll
                for (int g = 0; g < kG; ++g)
                    if (ok && J.te[g] <= J.tb[g]) {
                        ok = wait_poll(bar(L::kBarQ + g), qj & 1, ctl);
                        if (ok) mbar_arrive(bar(L::kBarQE + g));
                    }
                if (!ok) break;
                for (int j = 0; j <= J.nkv; ++j) {
                    const int tk = t + j, s = tk % kStages;
                    if (j < J.nkv) {
                        if (!wait_poll(bar(L::kBarKF + s), (tk / kStages) & 1, ctl)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const int jp = j - 1, tp = tk - 1, sp = (tp + kStages) % kStages;
                    if (jp >= 0 && !wait_poll(bar(L::kBarVF + sp), (tp / kStages) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kb = sK + s * L::NB * L::kKVBox;
                    const uint32_t vb = sV + sp * L::NB * L::kKVBox;
#pragma unroll
                    for (int g = 0; g < kG; ++g) {
                        const uint32_t tS = tmem + g * 256, tO = tS + 128;
                        if (ok && jp >= J.tb[g] && jp < J.te[g]) {
                            // O_g += P_g V: P_g sits in the first 64 columns of S_g
                            const int jl = jp - J.tb[g];
                            if (!wait_poll(bar(L::kBarP + g), (gt[g] + jl) & 1, ctl)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
#pragma unroll
                            for (int k = 0; k < kN / 16; ++k) {
                                const uint64_t bd = sdesc(vb + k * 2048, L::kKVBox, 1024);
                                tc_mma_ta(tO, tS + k * 8, bd, idesc_o, (jl > 0 || k > 0) ? 1u : 0u);
                            }
                            if (jp == J.te[g] - 1) tc_commit(bar(L::kBarPV + g));
                        }
                        if (ok && j < J.nkv && j >= J.tb[g] && j < J.te[g]) {
                            if (j == J.tb[g]) {
                                // Q_g of this job is in shared memory (TMA, or the
                                // softmax warps' cp.async gather: generic-proxy
                                // writes, ordered before the MMA's reads here)
                                if (!wait_poll(bar(L::kBarQ + g), qj & 1, ctl)) {
                                    ok = false;
                                    break;
                                }
                                if (MODE == kPast) fence_proxy_async();
                                tc_fence_after();
                            }
                            // S_g = Q_g K^T (runs after the PV above: same thread, in order)
                            const uint32_t qb = sQ + g * L::NB * L::kQBox;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint32_t off = (uint32_t)(k % 4) * 32;  // 16 dims = 32 B
                                const uint64_t ad = sdesc(qb + (k / 4) * L::kQBox + off, 16, 1024);
                                const uint64_t bd = sdesc(kb + (k / 4) * L::kKVBox + off, 16, 1024);
                                tc_mma(tS, ad, bd, idesc_s, k > 0);
                            }
                            tc_commit(bar(L::kBarS + g));
                            // the job's last S_g: Q_g may be replaced once it completes
                            if (j == J.te[g] - 1) tc_commit(bar(L::kBarQE + g));
                        }
                    }
                    if (!ok) break;
                    if (j < J.nkv) tc_commit(bar(L::kBarKE + s));
                    if (jp >= 0) tc_commit(bar(L::kBarVE + sp));
                }
                t += J.nkv;
                ++qj;
#pragma unroll
                for (int g = 0; g < kG; ++g) gt[g] += J.te[g] - J.tb[g];
                job = njob;
                J = NJ;
            }
            // every MMA this thread issued has finished before TMEM is freed
            tc_commit(bar(L::kBarDrain));
            drain_bar(bar(L::kBarDrain), 0, a.wait_limit);
        }
        __syncwarp();  // reconverge before the CTA barrier (bar.sync is per warp)
    } else {
        // ================= softmax + epilogue (warps 2..9) =================
        const int g = (warp - 2) >> 2;  // Q tile of this warp
        const int quarter = warp & 3;   // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int jrow = g * kM + row;  // row inside the job
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tSg = tmem + lane_off + g * 256;
        const uint32_t tOg = tSg + 128;
        const uint32_t sQg = sQ + g * L::NB * L::kQBox;
        const uint32_t stg = base + L::kStage + (uint32_t)(warp - 2) * L::kStageWarp;
        // past mode: this row's regroup entry (token << 5 | slot) in job J
        auto list_entry = [&](const Job &J) -> int {
            return (jrow < J.nrows) ? __ldg(a.list + J.lbeg + jrow) : 0;
        };
        // past mode: gather job J's rows of Q for tile g (cp.async, zero rows
        // past nrows); q_full[g] completes when every thread's copies landed
        // Each copy instruction moves 128 bytes of each of four rows: lane ->
        // (row r = it * 4 + lane / 8 of this warp's 32, 16-byte chunk lane % 8).
        auto gather = [&](const Job &J, int e) {
            const int ch = lane & 7;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                const int er = __shfl_sync(0xffffffffu, e, r);
                const bool valid = g * kM + quarter * 32 + r < J.nrows;
                const __nv_bfloat16 *src = a.q + ((size_t)(er >> kSlotBits) * H + J.h) * D + ch * 8;
                const uint32_t dst = sQg + (uint32_t)(quarter * 32 + r) * 128 +
                                     ((uint32_t)(ch ^ (r & 7)) << 4);
#pragma unroll
                for (int x = 0; x < L::NB; ++x)
                    cp_async16(dst + x * L::kQBox,
                               valid ? (const void *)(src + x * kBox) : (const void *)a.q, valid);
            }
            cp_async_arrive_noinc(bar(L::kBarQ + g));
        };
        int gt = 0, gj = 0, qj = 0;  // S/P tiles of tile g, jobs with rows in tile g, jobs
        bool ok = true;
        int job = blockIdx.x;
        Job J;
        while (job < njobs && !get_job<MODE, FUSE>(a, job, J)) job += gridDim.x;
        int entry = 0;  // this row's regroup entry in the current job, past mode
        if (MODE == kPast && job < njobs) {
            entry = list_entry(J);
            gather(J, entry);
        }
        int dn = 0;  // past mode: descriptors taken from the producer
        while (ok && job < njobs) {
            add_union_tiles<FUSE>(a, J);
            // the next job's descriptor, one job ahead (past mode: from the
            // producer), and this row's entry in it, loaded now and used after
            // the last tile
            int njob = job + gridDim.x;
            Job NJ;  // (own-block mode; the past mode reads it from its slot when needed)
            const Job *pnj = &NJ;
            if (MODE == kPast) {
                if (!__all_sync(0xffffffffu, wait_bar(bar(L::kBarDF + (dn & 1)), (dn >> 1) & 1, ctl))) {
                    ok = false;
                    break;
                }
                const uint8_t *slot = gmisc + L::kDesc + (dn & 1) * L::kDescSlot;
                pnj = reinterpret_cast<const Job *>(slot);
                njob = *reinterpret_cast<const int *>(slot + sizeof(Job));
            } else {
                while (njob < njobs && !get_job<MODE, FUSE>(a, njob, NJ)) njob += gridDim.x;
            }
            const int next_entry = (MODE == kPast && njob < njobs) ? list_entry(*pnj) : 0;
            const int seq0 = J.seq0, h = J.h;
            const bool row_valid = jrow < J.nrows;
            int row_tok = -1, slot = 0;
            if (MODE == kPast) {
                row_tok = entry >> kSlotBits;
                slot = entry & ((1 << kSlotBits) - 1);
            } else {
                row_tok = seq0 + J.r0 + jrow;
                // warm L2 with this row's past partials; the merge reads them only
                // after the last tile, so the fetch overlaps the attention loop
                if (row_valid && !a.dense && a.km1 > 0 && J.nu == 0) {
                    // every earlier block was a candidate, so the row holds
                    // min(topk - 1, its block index) partials, slots 0, 1, ...
                    const int npre = min(a.km1, (row_tok - seq0) / a.g.bs);
                    const size_t prow = (size_t)h * a.g.total + row_tok;  // head-major partials
                    for (int s2 = 0; s2 < npre; ++s2) {
                        const char *po = reinterpret_cast<const char *>(a.part_o + (prow * a.km1 + s2) * D);
#pragma unroll
                        for (int ln = 0; ln < D * 2; ln += 128)
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(po + ln));
                    }
                }
            }
            const int i_loc = row_tok - seq0;  // position inside the sequence
            // fused job: bit u = this row selected union block u
            unsigned row_bits = 0u;
            const int tpb = a.g.bs / kN;           // K/V tiles per block
            const int nut = FUSE ? J.nu * tpb : 0;  // union tiles of a fused job
            if (FUSE && J.nu > 0 && row_valid) {
                const int ci = i_loc / a.g.bs;
                const int32_t *sel = a.idx + ((size_t)row_tok * H + h) * a.topk;
                for (int s2 = 0; s2 < a.km1; ++s2) {
                    const int c = __ldg(sel + s2);
                    if (c < 0 || c >= ci) break;
                    for (int u = 0; u < J.nu; ++u)
                        if (__ldg(a.job_ub + job * kMaxUnion + u) == c) row_bits |= 1u << u;
                }
            }
            const int rb = (MODE == kCurrent && !a.dense) ? (i_loc / a.g.bs) * a.g.bs : 0;
            const int g_first = J.r0 + g * kM;
            const int g_last = min(J.r0 + (g + 1) * kM, J.r0 + J.nrows) - 1;
            const int rb_max = (MODE == kCurrent && !a.dense) ? (g_last / a.g.bs) * a.g.bs : 0;
            const int my_tb = (g == 0) ? J.tb[0] : J.tb[kG - 1];
            const int ntile = ((g == 0) ? J.te[0] : J.te[kG - 1]) - my_tb;
            const int kv_lo = J.kv_lo, kv_tok0 = J.kv_tok0, kv_end = J.kv_end;

            float m_run = -INFINITY, l_run = 0.f;
            int ucur = 0, usub = 0;  // union block and tile within it (fused jobs start at tile 0)
            for (int jl = 0; jl < ntile; ++jl) {
                const int j = my_tb + jl;
                // S_g(j) is ready; the commit behind it also covers PV_g(j-1), so
                // O_g is stable and P_g's columns are free
                const bool sready = jl == 0 ? boundary_wait<MODE>(bar(L::kBarS + g), (gt + jl) & 1, ctl)
                                            : wait_bar(bar(L::kBarS + g), (gt + jl) & 1, ctl);
                if (!__all_sync(0xffffffffu, sready)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // a fused job's union tiles come first: a full past block, off
                // for the rows that did not select it
                const bool uni = FUSE && j < nut;
                bool row_off = false;
                if (uni) {
                    row_off = !((row_bits >> ucur) & 1u);
                    if (++usub == tpb) {
                        usub = 0;
                        ++ucur;
                    }
                }
                const int jo = j - nut;            // own tile index
                const int key0 = kv_lo + jo * kN;  // sequence-local position of column 0
                const bool need_mask =
                    (MODE == kPast) ? (kv_tok0 + (j + 1) * kN > kv_end)
                    : uni           ? row_off
                                    : (key0 + kN - 1 > g_first || key0 < rb_max ||
                                       seq0 + key0 + kN > kv_end);
                // masked columns are set to -inf (raw fp32 bits) in place; only the
                // tiles on the diagonal / at the end of a block need it
                const int kt0 = kv_tok0 + jo * kN;  // token of column 0
#define MOBA_MASK64(SR, BASE)                                                         \
    if (need_mask) {                                                                  \
        _Pragma("unroll") for (int c = 0; c < 64; ++c) {                              \
            const int col = (BASE) + c;                                               \
            const int kp = key0 + col;                                                \
            if (uni || kt0 + col >= kv_end || (MODE == kCurrent && (kp > i_loc || kp < rb))) \
                SR[c >> 5][c & 31] = 0xff800000u;                                     \
        }                                                                             \
    }
                // One pass per 64-key half: the half's max decides the offset mu
                // (raised, to a whole number, only when the max exceeds it by more
                // than 8, so P <= 2^8 and every rescale is by an exact power of 2),
                // then p = 2^(s * scale - mu) from the same registers, as bf16
                // pairs (keys 2c, 2c+1 in column c) over the first 64 columns of
                // S: half h2 goes to columns 32*h2 .. 32*h2+31, already read when
                // h2 = 1 is written.  When the second half raises mu, the first
                // half's P in TMEM and the running O and l are rescaled.
                const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t sr[2][32];
                    tc_ld32(tSg + 64 * h2, sr[0]);
                    tc_ld32(tSg + 64 * h2 + 32, sr[1]);
                    tc_wait_ld();
                    MOBA_MASK64(sr, 64 * h2)
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 64; c += 8) {
                        mx[(c >> 3) & 3] = fmax3(mx[(c >> 3) & 3], __uint_as_float(sr[c >> 5][c & 31]),
                                                 __uint_as_float(sr[c >> 5][(c & 31) + 1]));
                        mx[(c >> 3) & 3] = fmax3(mx[(c >> 3) & 3], __uint_as_float(sr[c >> 5][(c & 31) + 2]),
                                                 __uint_as_float(sr[c >> 5][(c & 31) + 3]));
                        mx[(c >> 3) & 3] = fmax3(mx[(c >> 3) & 3], __uint_as_float(sr[c >> 5][(c & 31) + 4]),
                                                 __uint_as_float(sr[c >> 5][(c & 31) + 5]));
                        mx[(c >> 3) & 3] = fmax3(mx[(c >> 3) & 3], __uint_as_float(sr[c >> 5][(c & 31) + 6]),
                                                 __uint_as_float(sr[c >> 5][(c & 31) + 7]));
                    }
                    const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
                    const bool raise = mt > m_run + 8.f;  // always for the first finite max
                    const float m_new = raise ? ceilf(mt) : m_run;
                    if (__any_sync(0xffffffffu, raise && (jl > 0 || h2 > 0))) {
                        // 2^(old mu - new mu): 0 while nothing was accumulated yet
                        const float alpha = raise ? pow2_whole(m_run - m_new) : 1.f;
                        if (jl > 0) {  // O holds earlier tiles (this job's first PV overwrites it)
#pragma unroll
                            for (int c0 = 0; c0 < D; c0 += 16) {
                                uint32_t o[16];
                                tc_ld16(tOg + c0, o);
                                tc_wait_ld();
#pragma unroll
                                for (int c = 0; c < 16; ++c)
                                    o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                                tc_st16(tOg + c0, o);
                            }
                        }
                        if (h2 > 0) {  // the first half's P was made with the old mu
                            tc_wait_st();
#pragma unroll
                            for (int c0 = 0; c0 < 32; c0 += 16) {
                                uint32_t pw[16];
                                tc_ld16(tSg + c0, pw);
                                tc_wait_ld();
#pragma unroll
                                for (int c = 0; c < 16; ++c) {
                                    float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[c]));
                                    __nv_bfloat162 bb = __floats2bfloat162_rn(f.x * alpha, f.y * alpha);
                                    pw[c] = *reinterpret_cast<uint32_t *>(&bb);
                                }
                                tc_st16(tSg + c0, pw);
                            }
                        }
                    }
                    if (raise) {
                        l_run *= pow2_whole(m_run - m_new);
                        m_run = m_new;
                    }
                    const float mu = (m_run == -INFINITY) ? 0.f : m_run;
                    const float2 nmu2 = make_float2(-mu, -mu);
                    float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float2 x = ffma2(make_float2(__uint_as_float(sr[(2 * c) >> 5][(2 * c) & 31]),
                                                           __uint_as_float(sr[(2 * c + 1) >> 5][(2 * c + 1) & 31])),
                                               sc2, nmu2);
                        float2 pp;
                        pp.x = fast_exp2(x.x);
                        pp.y = fast_exp2(x.y);
                        ls[c & 1] = fadd2(ls[c & 1], pp);
                        __nv_bfloat162 bb = __floats2bfloat162_rn(pp.x, pp.y);
                        pk[c] = *reinterpret_cast<uint32_t *>(&bb);
                    }
                    tc_st32(tSg + 32 * h2, pk);
                    l_run += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
                }
#undef MOBA_MASK64
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kBarP + g));
            }
            if (!ok) break;
            gt += ntile;
            // in past mode the next job's Q rows are gathered as soon as the MMA
            // has released Q_g (this job's S_g MMAs are done): they land while
            // this job's epilogue runs, and the next job's S_g needs no wait
            // on the softmax warps
            if (MODE == kPast && njob < njobs) {
                if (!__all_sync(0xffffffffu, wait_bar(bar(L::kBarQE + g), qj & 1, ctl))) {
                    ok = false;
                    break;
                }
                ++qj;
                gather(*pnj, next_entry);
            }

            // ---------------- epilogue ----------------
            if (ntile > 0) {
                if (!__all_sync(0xffffffffu, boundary_wait<MODE>(bar(L::kBarPV + g), gj & 1, ctl))) {
                    ok = false;
                    break;
                }
                ++gj;
                tc_fence_after();
                const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
                const float lse2 = m_run + __log2f(l_run);
                if (MODE == kPast) {
                    // partials are head-major, [head][token][slot]: a later
                    // own-block job reads its rows' partials as one run
                    const size_t pslot = ((size_t)h * a.g.total + row_tok) * a.km1 + slot;
                    const unsigned long long my_dst =
                        reinterpret_cast<unsigned long long>(a.part_o + pslot * D);
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 64) {
                        // 64 columns of my row as bf16 (128 bytes) into the staging rows
                        uint32_t o[2][32];
                        tc_ld32(tOg + c0, o[0]);
                        tc_ld32(tOg + c0 + 32, o[1]);
                        tc_wait_ld();
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int col = ch * 8 + 2 * e;
                                __nv_bfloat162 bb = __floats2bfloat162_rn(
                                    __uint_as_float(o[col >> 5][col & 31]) * inv,
                                    __uint_as_float(o[(col + 1) >> 5][(col + 1) & 31]) * inv);
                                w[e] = *reinterpret_cast<uint32_t *>(&bb);
                            }
                            st_shared_v4(stg + lane * 128 + ((uint32_t)(ch ^ (lane & 7)) << 4), w[0],
                                         w[1], w[2], w[3]);
                        }
                        __syncwarp();
                        // lane -> (row it * 4 + lane / 8, chunk lane % 8): whole lines out
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int r = it * 4 + (lane >> 3), ch = lane & 7;
                            const unsigned long long d = __shfl_sync(0xffffffffu, my_dst, r);
                            const int v = __shfl_sync(0xffffffffu, (int)row_valid, r);
                            const uint4 val =
                                ld_shared_v4(stg + r * 128 + ((uint32_t)(ch ^ (r & 7)) << 4));
                            if (v)
                                *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(d) + c0 +
                                                           ch * 8) = val;
                        }
                        __syncwarp();
                    }
                    if (row_valid) a.part_lse[pslot] = lse2;
                } else {
                    // log-sum-exp merge with the row's past partials (slots in
                    // ascending block order; every earlier block was a candidate,
                    // so there are min(topk - 1, block index) of them)
                    const size_t rowid = (size_t)row_tok * H + h;
                    const size_t prow = (size_t)h * a.g.total + row_tok;  // head-major partials
                    int np = 0;
                    float mmax = lse2;
                    if (row_valid && !a.dense && a.km1 > 0 && J.nu == 0) {
                        np = min(a.km1, i_loc / a.g.bs);
                        for (int s2 = 0; s2 < np; ++s2)
                            mmax = fmaxf(mmax, __ldg(a.part_lse + prow * a.km1 + s2));
                    }
                    float w_cur = 1.f, wsum = 1.f;
                    if (np > 0) {
                        w_cur = fast_exp2(lse2 - mmax);
                        wsum = w_cur;
                        for (int s2 = 0; s2 < np; ++s2)
                            wsum += fast_exp2(__ldg(a.part_lse + prow * a.km1 + s2) - mmax);
                    }
                    const float iw = 1.f / wsum;
                    const float fcur = w_cur * inv * iw;
                    const int np_warp = __reduce_max_sync(0xffffffffu, np);
                    // 32 columns per pass; staging [slot pair][32 rows][64 B]; the
                    // copies map lane -> (row it * 8 + lane / 4, 16-byte chunk lane % 4)
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        tc_ld32(tOg + c0, o);
                        tc_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * fcur);
                        for (int s0 = 0; s0 < np_warp; s0 += 2) {
#pragma unroll
                            for (int it = 0; it < 4; ++it) {
                                const int r = it * 8 + (lane >> 2), q4 = lane & 3;
                                const unsigned long long prid =
                                    __shfl_sync(0xffffffffu, (unsigned long long)prow, r);
                                const int npr = __shfl_sync(0xffffffffu, np, r);
#pragma unroll
                                for (int ss = 0; ss < 2; ++ss) {
                                    const bool v = s0 + ss < npr;
                                    const __nv_bfloat16 *src =
                                        a.part_o + (prid * a.km1 + s0 + ss) * D + c0 + q4 * 8;
                                    cp_async16(stg + ss * 2048 + r * 64 +
                                                   ((uint32_t)(q4 ^ ((r >> 1) & 3)) << 4),
                                               v ? (const void *)src : (const void *)a.part_o, v);
                                }
                            }
                            cp_async_wait_all();
                            __syncwarp();
#pragma unroll
                            for (int ss = 0; ss < 2; ++ss) {
                                if (s0 + ss < np) {
                                    const float w =
                                        fast_exp2(__ldg(a.part_lse + prow * a.km1 + s0 + ss) - mmax) * iw;
#pragma unroll
                                    for (int q4 = 0; q4 < 4; ++q4) {
                                        const uint4 f =
                                            ld_shared_v4(stg + ss * 2048 + lane * 64 +
                                                         ((uint32_t)(q4 ^ ((lane >> 1) & 3)) << 4));
                                        const __nv_bfloat162 *b2 =
                                            reinterpret_cast<const __nv_bfloat162 *>(&f);
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            const float2 fv = __bfloat1622float2(b2[e]);
                                            const int col = q4 * 8 + 2 * e;
                                            o[col] = __float_as_uint(fmaf(w, fv.x, __uint_as_float(o[col])));
                                            o[col + 1] =
                                                __float_as_uint(fmaf(w, fv.y, __uint_as_float(o[col + 1])));
                                        }
                                    }
                                }
                            }
                            __syncwarp();
                        }
                        // bf16 result (64 bytes of my row) re-laid, then whole rows out
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int col = q4 * 8 + 2 * e;
                                __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(o[col]),
                                                                          __uint_as_float(o[col + 1]));
                                w[e] = *reinterpret_cast<uint32_t *>(&bb);
                            }
                            st_shared_v4(stg + lane * 64 + ((uint32_t)(q4 ^ ((lane >> 1) & 3)) << 4),
                                         w[0], w[1], w[2], w[3]);
                        }
                        __syncwarp();
#pragma unroll
                        for (int it = 0; it < 4; ++it) {
                            const int r = it * 8 + (lane >> 2), q4 = lane & 3;
                            const unsigned long long rid =
                                __shfl_sync(0xffffffffu, (unsigned long long)rowid, r);
                            const int v = __shfl_sync(0xffffffffu, (int)row_valid, r);
                            const uint4 val =
                                ld_shared_v4(stg + r * 64 + ((uint32_t)(q4 ^ ((r >> 1) & 3)) << 4));
                            if (v) *reinterpret_cast<uint4 *>(a.out + rid * D + c0 + q4 * 8) = val;
                        }
                        __syncwarp();
                    }
                    if (row_valid) {
                        const float lse_out = (np > 0) ? mmax + __log2f(wsum) : lse2;
                        const size_t li = a.fixed
                                              ? ((size_t)J.b * H + h) * a.S_fixed + i_loc
                                              : (size_t)h * a.g.total + row_tok;
                        a.lse[li] = lse_out * 0.69314718055994530942f;
                    }
                }
                // O_g has been read: the next job's first PV may overwrite it
                tc_fence_before();
            }
            job = njob;
            J = *pnj;
            entry = next_entry;
            if (MODE == kPast) {
                // the slot may take the descriptor after the next
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kBarDE + (dn & 1)));
                ++dn;
            }
        }
        cp_async_wait_all();  // no copy of ours may land after the exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [total][H][D] bf16 viewed as a 3-D tensor (D, H, total); box = 64 dims x 1
// head x `rows` tokens, 128-byte swizzle.
bool make_tma_3d(CUtensorMap *m, const void *ptr, int total, int H, int D, int rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_tile_rows() { return tc::kRows; }

static tc::Args make_tc_args(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             __nv_bfloat16 *out, float *lse) {
    tc::Args a;
    a.g.cu = ws.cu;
    a.g.blk_base = ws.blk_base;
    a.g.bad = ws.bad;
    a.g.num_seqs = p.num_seqs;
    a.g.total = p.total;
    a.g.H = p.H;
    a.g.D = p.D;
    a.g.bs = p.bs;
    a.q = q;
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
    a.job_list = ws.job_list;
    a.n_lists = p.NBcap * p.H;
    a.n_rtiles = (p.max_len + tc::kRows - 1) / tc::kRows;
    a.n_jobs = a.n_rtiles * p.num_seqs * p.H;
    a.part_o = ws.part_o;
    a.part_lse = ws.part_lse;
    a.fused = fusion_enabled(p) ? 1 : 0;
    a.any_fused = ws.counts ? ws.counts + (size_t)p.NBcap * p.H : nullptr;
    a.job_nu = ws.job_nu;
    a.job_ub = ws.job_ub;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)p.D));
    a.status = status_word();
    a.wait_limit = p.wait_limit;
    a.debug_flags = p.debug_flags;
    return a;
}

template <int D, int MODE, bool FUSE>
static cudaError_t launch_tc(const Plan &p, const tc::Args &a, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    if (!make_tma_3d(&mq, q, p.total, p.H, D, tc::kM) ||
        !make_tma_3d(&mk, k, p.total, p.H, D, tc::kN) ||
        !make_tma_3d(&mv, v, p.total, p.H, D, tc::kN))
        return cudaErrorInvalidValue;
    const int smem = tc::Smem<D>::kRequest;
    auto kern = tc::attn_tc_kernel<D, MODE, FUSE>;
    // The block needs all of its 320 threads resident (warp roles are fixed);
    // refuse to launch if the build's register use would not allow that.
    static int checked[2][2][2] = {};
    int &chk = checked[D == 128][MODE][FUSE ? 1 : 0];
    if (!chk) {
        cudaFuncAttributes fa;
        cudaError_t e0 = cudaFuncGetAttributes(&fa, kern);
        if (e0 != cudaSuccess) return e0;
        chk = (fa.numRegs <= tc::kRegLaunch && fa.maxThreadsPerBlock >= tc::kThreads) ? 1 : -1;
    }
    if (chk < 0) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (fewer when there are fewer own-block jobs)
    int ctas = sm_count();
    if (MODE == tc::kCurrent && a.n_jobs < ctas) ctas = a.n_jobs;
    const dim3 grid(ctas > 0 ? ctas : 1);
    kern<<<grid, tc::kThreads, smem, st>>>(mq, mk, mv, a);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attn_past_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st) {
    if (p.dense || p.km1 == 0) return cudaSuccess;
    auto a = make_tc_args(p, ws, q, nullptr, nullptr);
    return p.D == 64 ? launch_tc<64, tc::kPast, false>(p, a, q, k, v, st)
                     : launch_tc<128, tc::kPast, false>(p, a, q, k, v, st);
}

cudaError_t launch_attn_current_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                   const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                   __nv_bfloat16 *out, float *lse, cudaStream_t st) {
    auto a = make_tc_args(p, ws, q, out, lse);
    // with fusion possible, both variants are launched and the fusion test's
    // flag lets one of them run: the variant without union tiles keeps the
    // own-block kernel's speed when no job fused
    cudaError_t e = p.D == 64 ? launch_tc<64, tc::kCurrent, false>(p, a, q, k, v, st)
                              : launch_tc<128, tc::kCurrent, false>(p, a, q, k, v, st);
    if (e != cudaSuccess || !a.fused) return e;
    return p.D == 64 ? launch_tc<64, tc::kCurrent, true>(p, a, q, k, v, st)
                     : launch_tc<128, tc::kCurrent, true>(p, a, q, k, v, st);
}

}  // namespace moba
