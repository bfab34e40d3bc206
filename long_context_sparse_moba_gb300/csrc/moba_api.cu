// moba_api.cu -- the C ABI declared in include/moba.h: argument validation,
// scratch layout and the launch sequence of the MoBA forward pass.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "moba.h"
#include "moba_internal.cuh"

#define MOBA_EXPORT extern "C" __attribute__((visibility("default")))

namespace moba {

// [0] status word; [1..4] where the first timeout happened (barrier shared
// address, parity, block, thread)
__device__ int g_moba_status[8];

int *status_word() {
    static std::atomic<int *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    int *a = addr[dev].load(std::memory_order_relaxed);
    if (!a) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_moba_status) != cudaSuccess) return nullptr;
        a = static_cast<int *>(p);
        addr[dev].store(a, std::memory_order_relaxed);
    }
    return a;
}

static std::atomic<unsigned long long> g_launches{0};

int past_tile_rows(const Plan &p) { return p.attn_kind == 0 ? tc_tile_rows() : mma_tile_rows(); }
cudaError_t launch_attn_past(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                             const __nv_bfloat16 *k, const __nv_bfloat16 *v, cudaStream_t st) {
    return p.attn_kind == 0 ? launch_attn_past_tc(p, ws, q, k, v, st)
                            : launch_attn_past_mma(p, ws, q, k, v, st);
}
cudaError_t launch_attn_current(const Plan &p, const Workspace &ws, const __nv_bfloat16 *q,
                                const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                __nv_bfloat16 *out, float *lse, cudaStream_t st) {
    return p.attn_kind == 0 ? launch_attn_current_tc(p, ws, q, k, v, out, lse, st)
                            : launch_attn_current_mma(p, ws, q, k, v, out, lse, st);
}
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n); }

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Optional phase timing: the caller's CUDA events, recorded on the call's
// stream between the phases of a forward call (set-up, kpool, gate, regroup,
// attention over past blocks, attention over the own block + merge).
constexpr int kPhases = 6;

static void prof_mark(void *const *events, int phase, cudaStream_t st) {
    if (events && events[phase]) cudaEventRecord(static_cast<cudaEvent_t>(events[phase]), st);
}

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Rows of the tensor-core gate's list of rows left to its exact kernel: every
// gate CTA owns the rows of its 128-row units (padded tiles included).
static size_t need_list_rows(const Plan &p) {
    return (size_t)p.H * ((size_t)p.total + 128 * (size_t)p.num_seqs);
}

// The job table is sized for the smaller tile of the two attention kernels, so
// that the workspace size does not depend on the per-call kernel choice.
static size_t job_rows_min() {
    const int a = tc_tile_rows(), b = mma_tile_rows();
    return (size_t)(a < b ? a : b);
}

size_t workspace_bytes(const Plan &p, Workspace *ws, char *base, bool backward) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> void * {
        void *r = base ? static_cast<void *>(base + off) : nullptr;
        off = align256(off + bytes);
        return r;
    };
    Workspace w;
    std::memset(&w, 0, sizeof w);
    w.cu = static_cast<int *>(take(sizeof(int) * (p.num_seqs + 1)));
    w.blk_base = static_cast<int *>(take(sizeof(int) * (p.num_seqs + 1)));
    w.gtile = static_cast<int *>(take(sizeof(int) * (p.num_seqs + 1)));
    w.bad = static_cast<int *>(take(sizeof(int)));
    const bool gate = !p.dense && p.km1 > 0;
    if (gate) {
        const size_t N = (size_t)p.NBcap * p.H;
        const size_t rows = (size_t)p.total * p.H;
        w.kbar = static_cast<float *>(take(sizeof(float) * N * p.D));
        w.idx = static_cast<int32_t *>(take(sizeof(int32_t) * rows * p.topk));
        w.counts = static_cast<int *>(take(sizeof(int) * (N + 1)));
        w.need_count = static_cast<int *>(take(sizeof(int) * kMaxGateCtas));
        w.need_list = static_cast<unsigned long long *>(
            take(2 * sizeof(long long) * need_list_rows(p)));
        w.list_off = static_cast<int *>(take(sizeof(int) * (N + 1)));
        w.tile_off = static_cast<int *>(take(sizeof(int) * (N + 1)));
        w.job_list = static_cast<int *>(
            take(sizeof(int) * (rows * p.km1 / (size_t)job_rows_min() + N + 1)));
        w.kbhi = static_cast<__nv_bfloat16 *>(take(sizeof(__nv_bfloat16) * N * p.D));
        w.kblo = static_cast<__nv_bfloat16 *>(take(sizeof(__nv_bfloat16) * N * p.D));
        w.knorm = static_cast<float *>(take(sizeof(float) * N));
        w.list = static_cast<int *>(take(sizeof(int) * rows * p.km1));
        if (!backward) {
            const size_t jobs =
                (size_t)((p.max_len + kFuseRows - 1) / kFuseRows) * p.num_seqs * p.H;
            w.job_nu = static_cast<int *>(take(sizeof(int) * jobs));
            w.job_ub = static_cast<int *>(take(sizeof(int) * jobs * kMaxUnion));
            w.part_o =
                static_cast<__nv_bfloat16 *>(take(sizeof(__nv_bfloat16) * rows * p.km1 * p.D));
            w.part_lse = static_cast<float *>(take(sizeof(float) * rows * p.km1));
        }
    }
    if (backward) {
        const size_t rows = (size_t)p.total * p.H;
        w.dq_acc = static_cast<float *>(take(sizeof(float) * rows * p.D));
        w.delta = static_cast<float *>(take(sizeof(float) * rows));
        if (gate) {
            w.list_l2 = static_cast<float *>(take(sizeof(float) * rows * p.km1));
            w.list_dl = static_cast<float *>(take(sizeof(float) * rows * p.km1));
            w.cta_hist = static_cast<int *>(
                take(sizeof(int) * (size_t)stable_regroup_ctas(p) * p.NBcap * p.H));
        }
    }
    if (ws) *ws = w;
    return off;
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
static int make_plan(int num_seqs, long long total, int max_len, int H, int D, int bs, int topk,
                     bool fixed, Plan *p) {
    if (num_seqs < 1 || H < 1 || max_len < 1 || total < 1 || bs < 1 || topk < 1)
        return MOBA_ERR_INVALID_ARG;
    if (bs % 64 != 0) return MOBA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return MOBA_ERR_UNSUPPORTED;
    if (total >= kMaxTokens || num_seqs > 65535 || H > 65535) return MOBA_ERR_UNSUPPORTED;
    const long long n_max = (max_len + (long long)bs - 1) / bs;
    p->num_seqs = num_seqs;
    p->total = (int)total;
    p->max_len = max_len;
    p->H = H;
    p->D = D;
    p->bs = bs;
    p->topk = topk;
    p->fixed = fixed;
    p->pool = MOBA_POOL_MEAN;
    p->gate_kind = MOBA_GATE_TENSOR_CORES;
    p->attn_kind = MOBA_ATTN_TCGEN05;
    p->debug_flags = 0;
    p->wait_limit = kDefaultWaitLimit;
    p->schedule = MOBA_SCHEDULE_ADAPTIVE;
    p->idx_in = nullptr;
    p->dense = topk >= n_max;
    p->km1 = p->dense ? 0 : topk - 1;
    const long long nbcap = fixed ? (long long)num_seqs * n_max : total / bs + num_seqs;
    if (nbcap * H >= (1ll << 31)) return MOBA_ERR_UNSUPPORTED;
    p->NBcap = (int)nbcap;
    if (!p->dense && p->km1 > kMaxPastSlots) return MOBA_ERR_UNSUPPORTED;
    if (total * H * (long long)(p->km1 > 0 ? p->km1 : 1) >= (1ll << 31)) return MOBA_ERR_UNSUPPORTED;
    return MOBA_OK;
}

// Copies the caller's per-call options into the plan (NULL = defaults).
static int apply_options(const moba_options_t *o, Plan *p) {
    if (!o) return MOBA_OK;
    if (o->pooling != MOBA_POOL_MEAN && o->pooling != MOBA_POOL_MAX) return MOBA_ERR_INVALID_ARG;
    if (o->gate_kernel != MOBA_GATE_TENSOR_CORES && o->gate_kernel != MOBA_GATE_CUDA_CORES)
        return MOBA_ERR_INVALID_ARG;
    if (o->attn_kernel != MOBA_ATTN_TCGEN05 && o->attn_kernel != MOBA_ATTN_MMA_SYNC)
        return MOBA_ERR_INVALID_ARG;
    if (o->debug_flags < 0) return MOBA_ERR_INVALID_ARG;
    if (o->schedule != MOBA_SCHEDULE_ADAPTIVE && o->schedule != MOBA_SCHEDULE_BLOCK_MAJOR)
        return MOBA_ERR_INVALID_ARG;
    p->schedule = o->schedule;
    p->pool = o->pooling;
    p->gate_kind = o->gate_kernel;
    p->attn_kind = o->attn_kernel;
    p->debug_flags = o->debug_flags;
    p->wait_limit = o->wait_limit_cycles > 0 ? o->wait_limit_cycles : kDefaultWaitLimit;
    if (o->idx_in && (reinterpret_cast<uintptr_t>(o->idx_in) & 3)) return MOBA_ERR_INVALID_ARG;
    p->idx_in = o->idx_in;
    return MOBA_OK;
}

static int cuda_status(cudaError_t e);

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;

#define MOBA_TRY(expr)                                   \
    do {                                                 \
        cudaError_t _e = (expr);                         \
        if (_e != cudaSuccess) {                         \
            g_last_cuda_error = _e;                      \
            return MOBA_ERR_CUDA;                        \
        }                                                \
    } while (0)

// Events the forward waits for just before the phase that reads each input
// (moba_attn_fwd_host: the copies of k, q and v land while earlier phases run).
#ifndef MOBA_HOST_COPY_PARTS
#define MOBA_HOST_COPY_PARTS 1
#endif
struct InputWaits {
    cudaEvent_t k[MOBA_HOST_COPY_PARTS], q[MOBA_HOST_COPY_PARTS], v[MOBA_HOST_COPY_PARTS];
};
static cudaError_t wait_all(cudaStream_t st, const cudaEvent_t (&ev)[MOBA_HOST_COPY_PARTS]) {
    for (cudaEvent_t e : ev) {
        const cudaError_t r = cudaStreamWaitEvent(st, e, 0);
        if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
}

static int run_forward(const Plan &p, const int *cu_dev, const void *q, const void *k,
                       const void *v, void *out, float *lse, void *workspace, size_t ws_bytes,
                       const moba_options_t *opt, cudaStream_t st,
                       const InputWaits *iw = nullptr) {
    Workspace ws;
    const size_t need = workspace_bytes(p, &ws, static_cast<char *>(workspace));
    if (!workspace || ws_bytes < need) return MOBA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOBA_ERR_WORKSPACE;
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    void *const *ev = opt ? opt->phase_events : nullptr;
    int32_t *idx_out = opt ? opt->idx_out : nullptr;
    prof_mark(ev, 0, st);
    MOBA_TRY(launch_setup(p, cu_dev, ws, st));
    prof_mark(ev, 1, st);
    const bool gate = !p.dense && p.km1 > 0;
    // the selection goes straight to the caller's buffer when one is given
    if (gate && idx_out) ws.idx = idx_out;
    if (iw) MOBA_TRY(wait_all(st, iw->k));
    if (gate) MOBA_TRY(launch_kpool(p, ws, kb, ws.kbar, st));
    prof_mark(ev, 2, st);
    const bool tc_gate = p.gate_kind == MOBA_GATE_TENSOR_CORES && gate_tc_supported(p);
    if (iw) MOBA_TRY(wait_all(st, iw->q));
    if (gate) {
        // the per-list counts
        MOBA_TRY(cudaMemsetAsync(ws.counts, 0, sizeof(int) * ((size_t)p.NBcap * p.H + 1), st));
        if (tc_gate) {
            MOBA_TRY(launch_kbar_split(p, ws.kbar, ws.kbhi, ws.kblo, ws.knorm, st));
            MOBA_TRY(launch_gate_tc(p, ws, qb, ws.kbar, ws.kbhi, ws.kblo, ws.knorm, ws.idx,
                                    ws.counts, ws.need_list, ws.need_count, st));
        } else {
            MOBA_TRY(launch_gate(p, ws, qb, ws.kbar, ws.idx, st));
        }
    } else if (idx_out) {
        MOBA_TRY(launch_fill_idx(p, ws, idx_out, st));
    }
    prof_mark(ev, 3, st);
    const bool fuse = gate && fusion_enabled(p);
    if (fuse) MOBA_TRY(launch_union(p, ws, tc_gate, st));
    if (gate) MOBA_TRY(launch_regroup(p, ws, tc_gate, fuse, st));
    prof_mark(ev, 4, st);
    if (iw) MOBA_TRY(wait_all(st, iw->v));
    MOBA_TRY(launch_attn_past(p, ws, qb, kb, vb, st));
    prof_mark(ev, 5, st);
    MOBA_TRY(launch_attn_current(p, ws, qb, kb, vb, static_cast<__nv_bfloat16 *>(out), lse, st));
    prof_mark(ev, 6, st);
    return MOBA_OK;
}

// Backward: the forward's selection recomputed (same kernels, so the same
// selection), then the gradient kernels.
static int run_backward(const Plan &p, const int *cu_dev, const void *q, const void *k,
                        const void *v, const void *out, const float *lse, const void *dout,
                        void *dq, void *dk, void *dv, void *workspace, size_t ws_bytes,
                        cudaStream_t st) {
    Workspace ws;
    const size_t need = workspace_bytes(p, &ws, static_cast<char *>(workspace), true);
    if (!workspace || ws_bytes < need) return MOBA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOBA_ERR_WORKSPACE;
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    MOBA_TRY(launch_setup(p, cu_dev, ws, st));
    // delta first: the regroup writes it beside every list entry
    MOBA_TRY(launch_bwd_delta(p, ws, static_cast<const __nv_bfloat16 *>(out),
                              static_cast<const __nv_bfloat16 *>(dout), st));
    const bool gate = !p.dense && p.km1 > 0;
    const bool tc_gate = p.gate_kind == MOBA_GATE_TENSOR_CORES && gate_tc_supported(p);
    if (gate && p.idx_in) {
        // the forward's selection: regroup it as it is
        ws.idx = const_cast<int32_t *>(p.idx_in);
        MOBA_TRY(launch_regroup_stable(p, ws, lse, st));
    } else if (gate) {
        MOBA_TRY(launch_kpool(p, ws, kb, ws.kbar, st));
        MOBA_TRY(cudaMemsetAsync(ws.counts, 0, sizeof(int) * ((size_t)p.NBcap * p.H + 1), st));
        if (tc_gate) {
            MOBA_TRY(launch_kbar_split(p, ws.kbar, ws.kbhi, ws.kblo, ws.knorm, st));
            MOBA_TRY(launch_gate_tc(p, ws, qb, ws.kbar, ws.kbhi, ws.kblo, ws.knorm, ws.idx,
                                    ws.counts, ws.need_list, ws.need_count, st));
        } else {
            MOBA_TRY(launch_gate(p, ws, qb, ws.kbar, ws.idx, st));
        }
        MOBA_TRY(launch_regroup_stable(p, ws, lse, st));
    }
    MOBA_TRY(cudaMemsetAsync(ws.dq_acc, 0, sizeof(float) * (size_t)p.total * p.H * p.D, st));
    MOBA_TRY(launch_attn_bwd(p, ws, qb, kb, static_cast<const __nv_bfloat16 *>(v),
                             static_cast<const __nv_bfloat16 *>(out), lse,
                             static_cast<const __nv_bfloat16 *>(dout),
                             static_cast<__nv_bfloat16 *>(dq), static_cast<__nv_bfloat16 *>(dk),
                             static_cast<__nv_bfloat16 *>(dv), st));
    return MOBA_OK;
}

static int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOBA_OK;
    g_last_cuda_error = e;
    return MOBA_ERR_CUDA;
}

static bool misaligned(const void *p) { return reinterpret_cast<uintptr_t>(p) & 15; }

// Small scratch for the tables of the pooling / gate entry points.
static int with_tables(const Plan &p, const int *cu_dev, cudaStream_t st,
                       int (*body)(const Plan &, Workspace &, void *), void *ctx) {
    Workspace ws;
    std::memset(&ws, 0, sizeof ws);
    const size_t one = align256(sizeof(int) * (p.num_seqs + 1));
    void *mem = nullptr;
    if (cudaMallocAsync(&mem, 3 * one + 256, st) != cudaSuccess) return MOBA_ERR_CUDA;
    ws.cu = static_cast<int *>(mem);
    ws.blk_base = reinterpret_cast<int *>(static_cast<char *>(mem) + one);
    ws.gtile = reinterpret_cast<int *>(static_cast<char *>(mem) + 2 * one);
    ws.bad = reinterpret_cast<int *>(static_cast<char *>(mem) + 3 * one);
    int rc = cuda_status(launch_setup(p, cu_dev, ws, st));
    if (rc == MOBA_OK) rc = body(p, ws, ctx);
    if (cudaFreeAsync(mem, st) != cudaSuccess && rc == MOBA_OK) rc = MOBA_ERR_CUDA;
    return rc;
}

struct PoolCtx {
    const void *k;
    float *kbar;
    cudaStream_t st;
};
struct GateCtx {
    const void *q;
    const float *kbar;
    int32_t *idx;
    cudaStream_t st;
};

static int pool_run(const Plan &p, Workspace &ws, void *c) {
    auto *x = static_cast<PoolCtx *>(c);
    return cuda_status(
        launch_kpool(p, ws, static_cast<const __nv_bfloat16 *>(x->k), x->kbar, x->st));
}
static int gate_run(const Plan &p, Workspace &ws, void *c) {
    auto *x = static_cast<GateCtx *>(c);
    const auto *q = static_cast<const __nv_bfloat16 *>(x->q);
    if (p.gate_kind != MOBA_GATE_TENSOR_CORES || !gate_tc_supported(p))
        return cuda_status(launch_gate(p, ws, q, x->kbar, x->idx, x->st));
    // stream-ordered scratch: the bf16 split of the caller's kbar, the norms,
    // and the rows left to the exact kernel
    const size_t n = (size_t)p.NBcap * p.H * p.D;
    const size_t b_split = align256(2 * n * sizeof(__nv_bfloat16));
    const size_t b_norm = align256(sizeof(float) * p.NBcap * p.H);
    const size_t b_list = align256(2 * sizeof(long long) * need_list_rows(p));
    void *mem = nullptr;
    if (cudaMallocAsync(&mem, b_split + b_norm + b_list + sizeof(int) * kMaxGateCtas, x->st) !=
        cudaSuccess)
        return MOBA_ERR_CUDA;
    char *m = static_cast<char *>(mem);
    auto *hi = reinterpret_cast<__nv_bfloat16 *>(m);
    auto *nrm = reinterpret_cast<float *>(m + b_split);
    auto *list = reinterpret_cast<unsigned long long *>(m + b_split + b_norm);
    auto *cnt = reinterpret_cast<int *>(m + b_split + b_norm + b_list);
    int rc = cuda_status(launch_kbar_split(p, x->kbar, hi, hi + n, nrm, x->st));
    if (rc == MOBA_OK)
        rc = cuda_status(launch_gate_tc(p, ws, q, x->kbar, hi, hi + n, nrm, x->idx, nullptr,
                                        list, cnt, x->st));
    if (cudaFreeAsync(mem, x->st) != cudaSuccess && rc == MOBA_OK) rc = MOBA_ERR_CUDA;
    return rc;
}

}  // namespace moba

using namespace moba;

MOBA_EXPORT int moba_num_blocks(int len, int block_size) {
    if (len <= 0 || block_size <= 0) return 0;
    return (int)(((long long)len + block_size - 1) / block_size);
}

MOBA_EXPORT const char *moba_status_string(int code) {
    switch (code) {
        case MOBA_OK: return "MOBA_OK";
        case MOBA_ERR_INVALID_ARG: return "MOBA_ERR_INVALID_ARG";
        case MOBA_ERR_UNSUPPORTED: return "MOBA_ERR_UNSUPPORTED";
        case MOBA_ERR_CUDA: return "MOBA_ERR_CUDA";
        case MOBA_ERR_WORKSPACE: return "MOBA_ERR_WORKSPACE";
        case MOBA_ERR_TIMEOUT: return "MOBA_ERR_TIMEOUT";
        default: return "MOBA_ERR_UNKNOWN";
    }
}


// ---------------------------------------------------------------------------
// pooling and gate entry points
// ---------------------------------------------------------------------------
MOBA_EXPORT int moba_kpool_ex(const void *k, float *kbar, int B, int H, int S, int D,
                              int block_size, const moba_options_t *opt, void *stream) {
    if (!k || !kbar) return MOBA_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(B, (long long)B * S, S, H, D, block_size, 1, true, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    if (misaligned(k) || misaligned(kbar)) return MOBA_ERR_INVALID_ARG;
    PoolCtx c{k, kbar, static_cast<cudaStream_t>(stream)};
    return with_tables(p, nullptr, c.st, pool_run, &c);
}

MOBA_EXPORT int moba_kpool(const void *k, float *kbar, int B, int H, int S, int D, int block_size,
                           void *stream) {
    return moba_kpool_ex(k, kbar, B, H, S, D, block_size, nullptr, stream);
}

MOBA_EXPORT int moba_kpool_varlen_ex(const void *k, float *kbar, const int32_t *cu_seqlens,
                                     int num_seqs, int total_tokens, int H, int D, int block_size,
                                     const moba_options_t *opt, void *stream) {
    if (!k || !kbar || !cu_seqlens) return MOBA_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(num_seqs, total_tokens, total_tokens, H, D, block_size, 1, false, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    if (misaligned(k) || misaligned(kbar)) return MOBA_ERR_INVALID_ARG;
    PoolCtx c{k, kbar, static_cast<cudaStream_t>(stream)};
    return with_tables(p, cu_seqlens, c.st, pool_run, &c);
}

MOBA_EXPORT int moba_kpool_varlen(const void *k, float *kbar, const int32_t *cu_seqlens,
                                  int num_seqs, int total_tokens, int H, int D, int block_size,
                                  void *stream) {
    return moba_kpool_varlen_ex(k, kbar, cu_seqlens, num_seqs, total_tokens, H, D, block_size,
                                nullptr, stream);
}

MOBA_EXPORT int moba_gate_topk_ex(const void *q, const float *kbar, int32_t *idx, int B, int H,
                                  int S, int D, int block_size, int topk,
                                  const moba_options_t *opt, void *stream) {
    if (!q || !kbar || !idx) return MOBA_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    if (topk - 1 > kMaxPastSlots && !p.dense) return MOBA_ERR_UNSUPPORTED;
    if (misaligned(q) || misaligned(kbar)) return MOBA_ERR_INVALID_ARG;
    GateCtx c{q, kbar, idx, static_cast<cudaStream_t>(stream)};
    return with_tables(p, nullptr, c.st, gate_run, &c);
}

MOBA_EXPORT int moba_gate_topk(const void *q, const float *kbar, int32_t *idx, int B, int H, int S,
                               int D, int block_size, int topk, void *stream) {
    return moba_gate_topk_ex(q, kbar, idx, B, H, S, D, block_size, topk, nullptr, stream);
}

MOBA_EXPORT int moba_gate_topk_varlen_ex(const void *q, const float *kbar, int32_t *idx,
                                         const int32_t *cu_seqlens, int num_seqs,
                                         int total_tokens, int H, int D, int block_size, int topk,
                                         const moba_options_t *opt, void *stream) {
    if (!q || !kbar || !idx || !cu_seqlens) return MOBA_ERR_INVALID_ARG;
    Plan p;
    int rc = make_plan(num_seqs, total_tokens, total_tokens, H, D, block_size, topk, false, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    if (misaligned(q) || misaligned(kbar)) return MOBA_ERR_INVALID_ARG;
    GateCtx c{q, kbar, idx, static_cast<cudaStream_t>(stream)};
    return with_tables(p, cu_seqlens, c.st, gate_run, &c);
}

MOBA_EXPORT int moba_gate_topk_varlen(const void *q, const float *kbar, int32_t *idx,
                                      const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                                      int H, int D, int block_size, int topk, void *stream) {
    return moba_gate_topk_varlen_ex(q, kbar, idx, cu_seqlens, num_seqs, total_tokens, H, D,
                                    block_size, topk, nullptr, stream);
}

// ---------------------------------------------------------------------------
// forward entry points
// ---------------------------------------------------------------------------
MOBA_EXPORT size_t moba_attn_fwd_workspace_size(int B, int H, int S, int D, int block_size,
                                                int topk) {
    Plan p;
    if (make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p)) return 0;
    return workspace_bytes(p, nullptr, nullptr);
}

MOBA_EXPORT size_t moba_workspace_size(int B, int H, int S, int D, int block_size, int topk) {
    return moba_attn_fwd_workspace_size(B, H, S, D, block_size, topk);
}

MOBA_EXPORT size_t moba_attn_fwd_varlen_workspace_size(int num_seqs, int total_tokens,
                                                       int max_seqlen, int H, int D,
                                                       int block_size, int topk) {
    Plan p;
    if (make_plan(num_seqs, total_tokens, max_seqlen, H, D, block_size, topk, false, &p)) return 0;
    return workspace_bytes(p, nullptr, nullptr);
}

static int check_tensors(const void *q, const void *k, const void *v, const void *out,
                         const void *lse) {
    if (!q || !k || !v || !out || !lse) return MOBA_ERR_INVALID_ARG;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out))
        return MOBA_ERR_INVALID_ARG;
    return MOBA_OK;
}

static int check_options_buffers(const moba_options_t *opt) {
    if (opt && opt->idx_out && (reinterpret_cast<uintptr_t>(opt->idx_out) & 3))
        return MOBA_ERR_INVALID_ARG;
    return MOBA_OK;
}

// Runs the forward in the caller's workspace, or in scratch taken from
// cudaMallocAsync on the stream and released on it afterwards.
static int forward_any(const Plan &p, const int *cu, const void *q, const void *k, const void *v,
                       void *out, float *lse, const moba_options_t *opt, void *workspace,
                       size_t ws_bytes, cudaStream_t st) {
    if (workspace) return run_forward(p, cu, q, k, v, out, lse, workspace, ws_bytes, opt, st);
    const size_t bytes = workspace_bytes(p, nullptr, nullptr);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) return MOBA_ERR_CUDA;
    int rc = run_forward(p, cu, q, k, v, out, lse, ws, bytes, opt, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && rc == MOBA_OK) rc = MOBA_ERR_CUDA;
    return rc;
}

MOBA_EXPORT int moba_attn_fwd_ex(const void *q, const void *k, const void *v, void *out,
                                 float *lse, int B, int H, int S, int D, int block_size, int topk,
                                 const moba_options_t *opt, void *workspace,
                                 size_t workspace_bytes_, void *stream) {
    int rc = check_tensors(q, k, v, out, lse);
    if (rc || (rc = check_options_buffers(opt))) return rc;
    Plan p;
    rc = make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    return forward_any(p, nullptr, q, k, v, out, lse, opt, workspace, workspace_bytes_,
                       static_cast<cudaStream_t>(stream));
}

MOBA_EXPORT int moba_attn_fwd_ws(const void *q, const void *k, const void *v, void *out,
                                 float *lse, int B, int H, int S, int D, int block_size, int topk,
                                 void *workspace, size_t workspace_bytes_, void *stream) {
    if (!workspace) return MOBA_ERR_WORKSPACE;
    return moba_attn_fwd_ex(q, k, v, out, lse, B, H, S, D, block_size, topk, nullptr, workspace,
                            workspace_bytes_, stream);
}

MOBA_EXPORT int moba_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                              int B, int H, int S, int D, int block_size, int topk, void *stream) {
    return moba_attn_fwd_ex(q, k, v, out, lse, B, H, S, D, block_size, topk, nullptr, nullptr, 0,
                            stream);
}

// ---------------------------------------------------------------------------
// forward on host buffers: copies in, the forward, copies out, one call
// ---------------------------------------------------------------------------
// Device scratch: q, k, v, out (bf16), lse (fp32) and the forward's workspace,
// each from a 256-byte boundary.
struct HostScratch {
    size_t q, k, v, out, lse, ws, end;
};
static HostScratch host_scratch(const Plan &p) {
    HostScratch h;
    const size_t qkv = align256((size_t)p.total * p.H * p.D * 2);
    h.q = 0;
    h.k = h.q + qkv;
    h.v = h.k + qkv;
    h.out = h.v + qkv;
    h.lse = h.out + qkv;
    h.ws = h.lse + align256((size_t)p.total * p.H * 4);
    h.end = h.ws + workspace_bytes(p, nullptr, nullptr);
    return h;
}

MOBA_EXPORT size_t moba_attn_fwd_host_scratch_size(int B, int H, int S, int D, int block_size,
                                                   int topk) {
    Plan p;
    if (make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p) != MOBA_OK) return 0;
    return host_scratch(p).end;
}

// Copies a host range to or from the device in kCopyParts parts on as many
// streams, recording an event on each after its part.  One part: the host
// link, not the copy engines, bounds these copies (about 210 GB/s host to device
// measured with one, two or four streams alike).
constexpr int kCopyParts = MOBA_HOST_COPY_PARTS;
static cudaError_t copy_parts(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind,
                              const cudaStream_t (&cs)[kCopyParts],
                              cudaEvent_t (&done)[kCopyParts]) {
    const size_t part = (bytes / kCopyParts) & ~size_t(255);
    size_t off = 0;
    for (int i = 0; i < kCopyParts; ++i) {
        const size_t n = (i + 1 < kCopyParts) ? part : bytes - off;
        cudaError_t e = cudaSuccess;
        if (n)
            e = cudaMemcpyAsync(static_cast<char *>(dst) + off, static_cast<const char *>(src) + off,
                                n, kind, cs[i]);
        if (e == cudaSuccess) e = cudaEventRecord(done[i], cs[i]);
        if (e != cudaSuccess) return e;
        off += n;
    }
    return cudaSuccess;
}

MOBA_EXPORT int moba_attn_fwd_host(const void *q, const void *k, const void *v, void *out,
                                   float *lse, int B, int H, int S, int D, int block_size,
                                   int topk, const moba_options_t *opt, void *dev_scratch,
                                   size_t scratch_bytes, void *stream) {
    int rc = check_tensors(q, k, v, out, lse);
    if (rc || (rc = check_options_buffers(opt))) return rc;
    Plan p;
    rc = make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    const HostScratch hs = host_scratch(p);
    if (!dev_scratch || scratch_bytes < hs.end || (reinterpret_cast<uintptr_t>(dev_scratch) & 255))
        return MOBA_ERR_WORKSPACE;
    char *base = static_cast<char *>(dev_scratch);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qkv = (size_t)p.total * p.H * p.D * 2, lse_bytes = (size_t)p.total * p.H * 4;
    // the copy streams and their events, made for this call and released once
    // the work enqueued on them has run
    constexpr int P = kCopyParts;
    cudaStream_t cs[P];
    InputWaits iw;
    cudaEvent_t start = nullptr, fin = nullptr, back[P];
    cudaEvent_t *evs[2 + 4 * P];
    int nev = 0;
    evs[nev++] = &start;
    evs[nev++] = &fin;
    for (int i = 0; i < P; ++i) {
        cs[i] = nullptr;
        evs[nev++] = &back[i];
        evs[nev++] = &iw.k[i];
        evs[nev++] = &iw.q[i];
        evs[nev++] = &iw.v[i];
    }
    for (cudaEvent_t *e : evs) *e = nullptr;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < P && e == cudaSuccess; ++i)
        e = cudaStreamCreateWithFlags(&cs[i], cudaStreamNonBlocking);
    for (cudaEvent_t *ev : evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    // the copies in start after the caller's earlier work on its stream, in the
    // order the phases read them: k (pooling), q (gate), v (attention)
    if (e == cudaSuccess) e = cudaEventRecord(start, st);
    for (int i = 0; i < P && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(cs[i], start, 0);
    if (e == cudaSuccess) e = copy_parts(base + hs.k, k, qkv, cudaMemcpyHostToDevice, cs, iw.k);
    if (e == cudaSuccess) e = copy_parts(base + hs.q, q, qkv, cudaMemcpyHostToDevice, cs, iw.q);
    if (e == cudaSuccess) e = copy_parts(base + hs.v, v, qkv, cudaMemcpyHostToDevice, cs, iw.v);
    if (e == cudaSuccess) {
        rc = run_forward(p, nullptr, base + hs.q, base + hs.k, base + hs.v, base + hs.out,
                         reinterpret_cast<float *>(base + hs.lse), base + hs.ws, hs.end - hs.ws,
                         opt, st, &iw);
        // the results out, then the caller's stream waits for them
        if (rc == MOBA_OK) {
            e = cudaEventRecord(fin, st);
            for (int i = 0; i < P && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(cs[i], fin, 0);
            if (e == cudaSuccess)
                e = copy_parts(out, base + hs.out, qkv, cudaMemcpyDeviceToHost, cs, back);
            // lse is small: one copy on the first stream, after its part of out
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(lse, base + hs.lse, lse_bytes, cudaMemcpyDeviceToHost, cs[0]);
            if (e == cudaSuccess) e = cudaEventRecord(back[0], cs[0]);
            for (int i = 0; i < P && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(st, back[i], 0);
        }
    }
    for (cudaEvent_t *ev : evs)
        if (*ev) cudaEventDestroy(*ev);
    for (cudaStream_t c : cs)
        if (c) cudaStreamDestroy(c);
    if (rc != MOBA_OK) return rc;
    return cuda_status(e);
}

MOBA_EXPORT int moba_attn_fwd_varlen_ex(const void *q, const void *k, const void *v, void *out,
                                        float *lse, const int32_t *cu_seqlens, int num_seqs,
                                        int total_tokens, int max_seqlen, int H, int D,
                                        int block_size, int topk, const moba_options_t *opt,
                                        void *workspace, size_t workspace_bytes_, void *stream) {
    int rc = check_tensors(q, k, v, out, lse);
    if (rc || (rc = check_options_buffers(opt))) return rc;
    if (!cu_seqlens) return MOBA_ERR_INVALID_ARG;
    Plan p;
    rc = make_plan(num_seqs, total_tokens, max_seqlen, H, D, block_size, topk, false, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    return forward_any(p, cu_seqlens, q, k, v, out, lse, opt, workspace, workspace_bytes_,
                       static_cast<cudaStream_t>(stream));
}

MOBA_EXPORT int moba_attn_fwd_varlen_ws(const void *q, const void *k, const void *v, void *out,
                                        float *lse, const int32_t *cu_seqlens, int num_seqs,
                                        int total_tokens, int max_seqlen, int H, int D,
                                        int block_size, int topk, void *workspace,
                                        size_t workspace_bytes_, void *stream) {
    if (!workspace) return MOBA_ERR_WORKSPACE;
    return moba_attn_fwd_varlen_ex(q, k, v, out, lse, cu_seqlens, num_seqs, total_tokens,
                                   max_seqlen, H, D, block_size, topk, nullptr, workspace,
                                   workspace_bytes_, stream);
}

MOBA_EXPORT int moba_attn_fwd_varlen(const void *q, const void *k, const void *v, void *out,
                                     float *lse, const int32_t *cu_seqlens, int num_seqs,
                                     int total_tokens, int max_seqlen, int H, int D,
                                     int block_size, int topk, void *stream) {
    return moba_attn_fwd_varlen_ex(q, k, v, out, lse, cu_seqlens, num_seqs, total_tokens,
                                   max_seqlen, H, D, block_size, topk, nullptr, nullptr, 0, stream);
}

// ---------------------------------------------------------------------------
// backward entry points
// ---------------------------------------------------------------------------
static int check_bwd_tensors(const void *q, const void *k, const void *v, const void *out,
                             const float *lse, const void *dout, const void *dq, const void *dk,
                             const void *dv) {
    int rc = check_tensors(q, k, v, out, lse);
    if (rc) return rc;
    if (!dout || !dq || !dk || !dv) return MOBA_ERR_INVALID_ARG;
    if (misaligned(dout) || misaligned(dq) || misaligned(dk) || misaligned(dv))
        return MOBA_ERR_INVALID_ARG;
    return MOBA_OK;
}

MOBA_EXPORT size_t moba_attn_bwd_workspace_size(int B, int H, int S, int D, int block_size,
                                                int topk) {
    Plan p;
    if (make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p)) return 0;
    return workspace_bytes(p, nullptr, nullptr, true);
}

MOBA_EXPORT size_t moba_attn_bwd_varlen_workspace_size(int num_seqs, int total_tokens,
                                                       int max_seqlen, int H, int D,
                                                       int block_size, int topk) {
    Plan p;
    if (make_plan(num_seqs, total_tokens, max_seqlen, H, D, block_size, topk, false, &p)) return 0;
    return workspace_bytes(p, nullptr, nullptr, true);
}

static int backward_any(const Plan &p, const int *cu, const void *q, const void *k, const void *v,
                        const void *out, const float *lse, const void *dout, void *dq, void *dk,
                        void *dv, void *workspace, size_t ws_bytes, cudaStream_t st) {
    if (workspace)
        return run_backward(p, cu, q, k, v, out, lse, dout, dq, dk, dv, workspace, ws_bytes, st);
    const size_t bytes = workspace_bytes(p, nullptr, nullptr, true);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, st) != cudaSuccess) return MOBA_ERR_CUDA;
    int rc = run_backward(p, cu, q, k, v, out, lse, dout, dq, dk, dv, ws, bytes, st);
    if (cudaFreeAsync(ws, st) != cudaSuccess && rc == MOBA_OK) rc = MOBA_ERR_CUDA;
    return rc;
}

MOBA_EXPORT int moba_attn_bwd_ex(const void *q, const void *k, const void *v, const void *out,
                                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                 int B, int H, int S, int D, int block_size, int topk,
                                 const moba_options_t *opt, void *workspace,
                                 size_t workspace_bytes_, void *stream) {
    int rc = check_bwd_tensors(q, k, v, out, lse, dout, dq, dk, dv);
    if (rc) return rc;
    Plan p;
    rc = make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    return backward_any(p, nullptr, q, k, v, out, lse, dout, dq, dk, dv, workspace,
                        workspace_bytes_, static_cast<cudaStream_t>(stream));
}

MOBA_EXPORT int moba_attn_bwd_ws(const void *q, const void *k, const void *v, const void *out,
                                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                 int B, int H, int S, int D, int block_size, int topk,
                                 void *workspace, size_t workspace_bytes_, void *stream) {
    if (!workspace) return MOBA_ERR_WORKSPACE;
    return moba_attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, H, S, D, block_size, topk,
                            nullptr, workspace, workspace_bytes_, stream);
}

MOBA_EXPORT int moba_attn_bwd(const void *q, const void *k, const void *v, const void *out,
                              const float *lse, const void *dout, void *dq, void *dk, void *dv,
                              int B, int H, int S, int D, int block_size, int topk, void *stream) {
    return moba_attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, B, H, S, D, block_size, topk,
                            nullptr, nullptr, 0, stream);
}

MOBA_EXPORT int moba_attn_bwd_varlen_ex(const void *q, const void *k, const void *v,
                                        const void *out, const float *lse, const void *dout,
                                        void *dq, void *dk, void *dv, const int32_t *cu_seqlens,
                                        int num_seqs, int total_tokens, int max_seqlen, int H,
                                        int D, int block_size, int topk,
                                        const moba_options_t *opt, void *workspace,
                                        size_t workspace_bytes_, void *stream) {
    int rc = check_bwd_tensors(q, k, v, out, lse, dout, dq, dk, dv);
    if (rc) return rc;
    if (!cu_seqlens) return MOBA_ERR_INVALID_ARG;
    Plan p;
    rc = make_plan(num_seqs, total_tokens, max_seqlen, H, D, block_size, topk, false, &p);
    if (rc || (rc = apply_options(opt, &p))) return rc;
    return backward_any(p, cu_seqlens, q, k, v, out, lse, dout, dq, dk, dv, workspace,
                        workspace_bytes_, static_cast<cudaStream_t>(stream));
}

MOBA_EXPORT int moba_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *out,
                                     const float *lse, const void *dout, void *dq, void *dk,
                                     void *dv, const int32_t *cu_seqlens, int num_seqs,
                                     int total_tokens, int max_seqlen, int H, int D,
                                     int block_size, int topk, void *stream) {
    return moba_attn_bwd_varlen_ex(q, k, v, out, lse, dout, dq, dk, dv, cu_seqlens, num_seqs,
                                   total_tokens, max_seqlen, H, D, block_size, topk, nullptr,
                                   nullptr, 0, stream);
}

// ---------------------------------------------------------------------------
// status, tally
// ---------------------------------------------------------------------------
static thread_local int g_last_timeout[4] = {0, 0, 0, 0};

MOBA_EXPORT void moba_debug_timeout_info(int *out4) {
    if (out4)
        for (int i = 0; i < 4; ++i) out4[i] = g_last_timeout[i];
}

MOBA_EXPORT int moba_get_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOBA_ERR_CUDA;
    int v[8];
    if (cudaMemcpyFromSymbol(v, g_moba_status, sizeof v) != cudaSuccess) return MOBA_ERR_CUDA;
    for (int i = 0; i < 4; ++i) g_last_timeout[i] = v[1 + i];
    const int zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_moba_status, zero, sizeof zero) != cudaSuccess) return MOBA_ERR_CUDA;
    return v[0];
}

MOBA_EXPORT unsigned long long moba_launch_count(void) { return g_launches.load(); }

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
static int decode_check(const void *q, const void *k, const void *v, const float *kbar,
                        const int32_t *lens, const void *out, const float *lse, int B, int H,
                        int S_max, int D, int bs, int topk) {
    if (!q || !k || !v || !kbar || !lens || !out || !lse) return MOBA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || S_max < 1 || bs < 1 || bs % 64 != 0 || topk < 1)
        return MOBA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return MOBA_ERR_UNSUPPORTED;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(kbar))
        return MOBA_ERR_INVALID_ARG;
    const long long n_max = ((long long)S_max + bs - 1) / bs;
    // a scored row keeps its top list in registers
    if (topk - 1 > decode_km1_max() && topk < n_max) return MOBA_ERR_UNSUPPORTED;
    if ((long long)B * H * topk >= (1ll << 31) || (long long)B * n_max * H >= (1ll << 31))
        return MOBA_ERR_UNSUPPORTED;
    return MOBA_OK;
}

MOBA_EXPORT size_t moba_decode_workspace_size(int B, int H, int D, int topk) {
    if (B < 1 || H < 1 || (D != 64 && D != 128) || topk < 1) return 0;
    return decode_scratch(nullptr, B, H, D, topk, nullptr, nullptr, nullptr, nullptr);
}

MOBA_EXPORT int moba_decode_fwd_ws(const void *q, const void *k_cache, const void *v_cache,
                                   const float *kbar, const int32_t *cache_lens, void *out,
                                   float *lse, int32_t *idx, int B, int H, int S_max, int D,
                                   int block_size, int topk, void *workspace,
                                   size_t workspace_bytes_, void *stream) {
    int rc = decode_check(q, k_cache, v_cache, kbar, cache_lens, out, lse, B, H, S_max, D,
                          block_size, topk);
    if (rc) return rc;
    const size_t need = decode_scratch(nullptr, B, H, D, topk, nullptr, nullptr, nullptr, nullptr);
    if (!workspace || workspace_bytes_ < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return MOBA_ERR_WORKSPACE;
    auto st = static_cast<cudaStream_t>(stream);
    const size_t toff = decode_ticket_offset(B, H, D, topk);
    MOBA_TRY(cudaMemsetAsync(static_cast<char *>(workspace) + toff, 0, sizeof(int) * (size_t)B * H,
                             st));
    return cuda_status(launch_decode(q, k_cache, v_cache, kbar, cache_lens, out, lse, idx, B, H,
                                     S_max, D, block_size, topk, workspace, st));
}

MOBA_EXPORT int moba_decode_fwd(const void *q, const void *k_cache, const void *v_cache,
                                const float *kbar, const int32_t *cache_lens, void *out,
                                float *lse, int32_t *idx, int B, int H, int S_max, int D,
                                int block_size, int topk, void *stream) {
    int rc = decode_check(q, k_cache, v_cache, kbar, cache_lens, out, lse, B, H, S_max, D,
                          block_size, topk);
    if (rc) return rc;
    auto st = static_cast<cudaStream_t>(stream);
    const size_t bytes = decode_scratch(nullptr, B, H, D, topk, nullptr, nullptr, nullptr, nullptr);
    void *mem = nullptr;
    if (cudaMallocAsync(&mem, bytes, st) != cudaSuccess) return MOBA_ERR_CUDA;
    rc = moba_decode_fwd_ws(q, k_cache, v_cache, kbar, cache_lens, out, lse, idx, B, H, S_max, D,
                            block_size, topk, mem, bytes, stream);
    if (cudaFreeAsync(mem, st) != cudaSuccess && rc == MOBA_OK) rc = MOBA_ERR_CUDA;
    return rc;
}

// ---------------------------------------------------------------------------
// Forward pass that allocates nothing.  Its scratch lives in one file-scope
// device array that every device loading this library keeps until the process
// exits.  Host code only sees a stand-in for the array's name, so the device
// address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
static constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

static void *static_scratch() {
    static std::atomic<void *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *a = addr[dev].load(std::memory_order_relaxed);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev].store(a, std::memory_order_relaxed);
    }
    return a;
}

MOBA_EXPORT size_t moba_attn_fwd_noalloc_capacity(void) { return kStaticScratchBytes; }

MOBA_EXPORT int moba_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                                      float *lse, int B, int H, int S, int D, int block_size,
                                      int topk, void *stream) {
    int rc = check_tensors(q, k, v, out, lse);
    if (rc) return rc;
    Plan p;
    rc = make_plan(B, (long long)B * S, S, H, D, block_size, topk, true, &p);
    if (rc) return rc;
    if (workspace_bytes(p, nullptr, nullptr) > kStaticScratchBytes) return MOBA_ERR_WORKSPACE;
    void *scratch = static_scratch();
    if (!scratch) return MOBA_ERR_CUDA;
    // run_forward clears the per-(block, head) counters itself (a memset, not
    // an allocation); every other scratch area is written before it is read
    return run_forward(p, nullptr, q, k, v, out, lse, scratch, kStaticScratchBytes, nullptr,
                       static_cast<cudaStream_t>(stream));
}

MOBA_EXPORT const char *moba_last_cuda_error(void) {
    return cudaGetErrorString(g_last_cuda_error);
}
