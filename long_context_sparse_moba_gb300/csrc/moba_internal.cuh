// moba_internal.cuh -- shared definitions of the MoBA sm_103a kernels.
//
// Geometry: sequences are packed token-major ([token][H][D]); a fixed-length
// batch [B][S][H][D] is the packed case with cu_seqlens = {0, S, 2S, ...}.
// Every kernel reads the per-sequence tables built by moba_setup_kernel:
//   cu[b]        first token of sequence b (cu[num_seqs] = total tokens)
//   blk_base[b]  global id of block 0 of sequence b (blk_base[num_seqs] = NB)
// Global block g of sequence b, local block c: g = blk_base[b] + c.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moba {

constexpr int kMaxPastSlots = 31;      // topk - 1 limit when gating is needed
constexpr int kSlotBits = 5;           // regroup entry = token << 5 | slot
constexpr int kMaxTokens = 1 << 26;
constexpr int kMaxGateCtas = 1024;     // CTAs of the tensor-core gate at most
// query-major fusion of the own-block jobs (256 rows of one block and head)
constexpr int kFuseRows = 256;         // rows per own-block job
constexpr int kMaxUnion = 8;           // past blocks a fused job may visit

// Device status word of the current device (defined in moba_api.cu); kernels
// with bounded waits record MOBA_ERR_TIMEOUT there.  moba_get_status reads
// and clears it.
int *status_word();

struct Geometry {
    const int *cu;        // [num_seqs + 1]
    const int *blk_base;  // [num_seqs + 1]
    // set by the table set-up when caller-provided sequence offsets are
    // inconsistent (not starting at 0, decreasing, longer than max_seqlen, or
    // not ending at total); every kernel that reads the tables returns at once
    const int *bad;
    int num_seqs;
    int total;            // tokens
    int H, D, bs;
};

// Largest b in [0, num_seqs) with tab[b] <= x (tab ascending, tab[0] = 0).
__device__ __forceinline__ int upper_index(const int *__restrict__ tab, int num_seqs, int x) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(tab + mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Scratch carved out of one workspace allocation (offsets 256-byte aligned).
struct Workspace {
    int *cu;          // [num_seqs + 1]
    int *blk_base;    // [num_seqs + 1]
    int *gtile;       // [num_seqs + 1]  128-row gate tiles before each sequence
    int *bad;         // [1] inconsistent sequence offsets (see Geometry::bad)
    float *kbar;      // [NBcap][H][D]
    int32_t *idx;     // [total][H][topk]
    int *counts;      // [NBcap * H]   queries per (block, head) past list (zero
                      //               again once the scatter has used them),
                      //               then one word: some own-block job fused
    int *need_count;  // [kMaxGateCtas] rows each tensor-core gate CTA left to the exact kernel
    unsigned long long *need_list;  // [2 * total * H] those rows and their candidates
    int *list_off;    // [NBcap * H + 1]
    int *tile_off;    // [NBcap * H + 1]  first attention job of each list
    int *job_list;    // [jobs]  list of every past-block attention job
    __nv_bfloat16 *kbhi, *kblo;  // [NBcap][H][D] bf16 split of kbar (tensor-core gate)
    float *knorm;                // [NBcap][H] L2 norm of each pooled key
    int *list;        // [total * H * km1]  entries token << 5 | slot
    int *job_nu;      // [own-block jobs]  past blocks of a fused job (0: not fused)
    int *job_ub;      // [own-block jobs][kMaxUnion]  those blocks, ascending
    __nv_bfloat16 *part_o;  // [H][total][km1][D]  normalised partial outputs (bf16), head-major
    float *part_lse;  // [H][total][km1]     partial log2-sum-exp
    // backward pass only (part_o / part_lse are not carved then)
    float *dq_acc;    // [total][H][D]  fp32 dq accumulator
    float *delta;     // [H][total]     dO . O per row
    float *list_l2, *list_dl;  // [total * H * km1] lse (log2) and dO . O of each list entry's row
    int *cta_hist;    // [stable regroup CTAs][NBcap * H]  selections per CTA and list
};

struct Plan {
    int num_seqs, total, max_len, H, D, bs, topk;
    int NBcap;        // upper bound of the global block count
    int km1;          // past slots per row (topk - 1), 0 on the dense path
    bool dense;       // topk covers every block of every sequence
    bool fixed;       // [B][S] layout (lse [B][H][S]) rather than varlen
    // per-call options (moba_options_t); defaults are all zero except the wait
    int pool;               // key pooling: 0 mean, 1 element-wise max
    int gate_kind;          // 0 tensor-core scores + exact candidates, 1 CUDA cores
    int attn_kind;          // 0 tcgen05 / TMEM / TMA, 1 warp-level mma.sync
    int debug_flags;        // bit 0: the K/V producer skips its first load
    long long wait_limit;   // clock64 budget of one bounded wait
    int schedule;           // 0 adaptive (fused own-block jobs where it pays), 1 block-major
    const int32_t *idx_in;  // backward: the forward's selection, or nullptr (recompute)
};

// clock64 budget of one bounded wait when the caller gives none (~2 s at 2 GHz)
constexpr long long kDefaultWaitLimit = 4000000000ll;

// Returns from a kernel when the table set-up flagged the caller's sequence
// offsets; every thread of the kernel reads the same word, so the whole grid
// leaves before any barrier.
#define MOBA_RETURN_IF_BAD(g)                 \
    do {                                      \
        if ((g).bad && *(g).bad) return;      \
    } while (0)

// backward = true: the backward pass's scratch (no partial outputs; the dq
// accumulator and the per-row dO . O instead)
size_t workspace_bytes(const Plan &p, Workspace *ws, char *base, bool backward = false);

// ---- launchers (each returns cudaGetLastError() of its launch) ----
cudaError_t launch_setup(const Plan &p, const int *cu_dev, Workspace &ws, cudaStream_t st);
cudaError_t launch_kpool(const Plan &p, const Workspace &ws, const __nv_bfloat16 *k,
                         float *kbar, cudaStream_t st);
cudaError_t launch_gate(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                        const float *kbar, int32_t *idx, cudaStream_t st);
// Own-block jobs (256-row tiles x of a sequence) run heavy (late) tiles
// first: job id = ((n_rtiles - 1 - x) * num_seqs + b) * H + h.
// Query-major fusion: an own-block job (256 rows of one block and head) whose
// rows all chose the same topk - 1 past blocks (among more candidates than
// that) attends to those blocks itself, so its rows leave the regroup lists
// and write no partial outputs.  Available with the tcgen05 attention, block
// sizes that are multiples of 256 and topk <= 9.
bool fusion_enabled(const Plan &p);
// the own-block jobs' unions of past selections (ws.job_nu, ws.job_ub); with
// counted, the fused rows' selections are taken back out of ws.counts
cudaError_t launch_union(const Plan &p, const Workspace &ws, bool counted, cudaStream_t st);
// per-(block, head) lists of the past selections: count (unless the gate has
// already added its selections into ws.counts), scan, scatter; with
// skip_fused, the rows of fused own-block jobs are left out
cudaError_t launch_regroup(const Plan &p, const Workspace &ws, bool counted, bool skip_fused,
                           cudaStream_t st);
// the same lists with their entries in an order fixed by the selection alone
// (every call places them alike); needs ws.cta_hist, rewrites ws.counts.  With
// lse (the forward's, its layout per the plan) and ws.delta, each entry's
// row lse (log2) and delta go into ws.list_l2 / ws.list_dl beside it.
cudaError_t launch_regroup_stable(const Plan &p, const Workspace &ws, const float *lse,
                                  cudaStream_t st);
// delta = dO . O per row into ws.delta ([H][total])
cudaError_t launch_bwd_delta(const Plan &p, const Workspace &ws, const __nv_bfloat16 *out,
                             const __nv_bfloat16 *dout, cudaStream_t st);
// CTAs of the stable regroup (rows of ws.cta_hist)
int stable_regroup_ctas(const Plan &p);
// attention over the selected past blocks (skipped on the dense / top-1 paths)
cudaError_t launch_attn_past(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st);
// causal attention inside the own block (every earlier key on the dense path)
// merged with the past partials
cudaError_t launch_attn_current(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                __nv_bfloat16 *out, float *lse, cudaStream_t st);

// count of kernels this library has launched (for the benchmark's launch tally)
void note_launches(int n);

// streaming multiprocessors of the current device (cached per device)
int sm_count();

// rows per tile of the past-block attention kernel the plan uses (regroup tiling)
int past_tile_rows(const Plan &p);

// the two attention implementations: tcgen05 / TMEM / TMA (default) and the
// warp-level mma.sync baseline
cudaError_t launch_attn_past_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st);
cudaError_t launch_attn_current_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                   const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                   __nv_bfloat16 *out, float *lse, cudaStream_t st);
cudaError_t launch_attn_past_mma(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                 const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st);
cudaError_t launch_attn_current_mma(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                    const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                    __nv_bfloat16 *out, float *lse, cudaStream_t st);
int tc_tile_rows();
// [total][H][D] bf16 as a 3-D TMA tensor (D, H, total), box 64 x 1 x rows, 128B swizzle
bool make_tma_3d(CUtensorMap *m, const void *ptr, int total, int H, int D, int rows);
// kbar (fp32) -> hi = bf16(kbar), lo = bf16(kbar - hi)
cudaError_t launch_kbar_split(const Plan &p, const float *kbar, __nv_bfloat16 *hi,
                              __nv_bfloat16 *lo, float *norm, cudaStream_t st);
// tensor-core gate (scores on tcgen05, exact fp32 re-score of the candidates);
// with counts != nullptr it also adds every past selection into counts.
// need_list (room for every row) and need_count (kMaxGateCtas ints, written by
// the gate) carry the rows whose selection the score margin cannot settle to
// the exact follow-up kernel
bool gate_tc_supported(const Plan &p);
cudaError_t launch_gate_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                           const float *kbar, const __nv_bfloat16 *khi, const __nv_bfloat16 *klo,
                           const float *knorm, int32_t *idx, int *counts,
                           unsigned long long *need_list,
                           int *need_count, cudaStream_t st);
int mma_tile_rows();
// decode: one query row per (sequence, head) against its KV cache
int decode_km1_max();
size_t decode_scratch(void *base, int B, int H, int D, int topk, int32_t **sel, float **ml,
                      float **po, int **ticket);
size_t decode_ticket_offset(int B, int H, int D, int topk);
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *kbar,
                          const int32_t *lens, void *out, float *lse, int32_t *idx, int B, int H,
                          int S_max, int D, int bs, int topk, void *scratch, cudaStream_t st);
// backward dk, dv and dq accumulation on the tcgen05 tensor cores (head size
// 128 with the tcgen05 attention kernels selected); ws.delta must hold dO . O
// and ws.dq_acc must be zero
bool bwd_tc_supported(const Plan &p);
cudaError_t launch_bwd_kv_tc(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                             const float *lse, const __nv_bfloat16 *dout, __nv_bfloat16 *dk,
                             __nv_bfloat16 *dv, cudaStream_t st);
// idx of the rows the gate does not run for (top-1, or top-k covering every
// block): the own block and every earlier one, ascending, -1 padded
cudaError_t launch_fill_idx(const Plan &p, const Workspace &ws, int32_t *idx, cudaStream_t st);
// backward: delta, then dk / dv (and the dq accumulator, which must be zero on
// entry) over the regroup lists, then dq
cudaError_t launch_attn_bwd(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                            const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                            const __nv_bfloat16 *out, const float *lse,
                            const __nv_bfloat16 *dout, __nv_bfloat16 *dq, __nv_bfloat16 *dk,
                            __nv_bfloat16 *dv, cudaStream_t st);

}  // namespace moba
