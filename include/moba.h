/*
 * moba.h -- C ABI of the MoBA (Mixture of Block Attention) forward pass on
 * GB300 (sm_103a).
 *
 * The method (pages cited by title and section):
 *   "Moonshot MoBA paper explained" (gsyq.cn/news/227272) section 3.1: the
 *     context is cut into blocks of block_size tokens; a block is represented
 *     by the mean of its keys; the gate scores blocks by that mean and masks
 *     future blocks; each query keeps top_k blocks (section 4.1 sorts the
 *     block scores and keeps the first top_k).
 *   "MOBA mixture of block attention for server-side long context"
 *     (hncyxsy.com/news/197418) section 3: the current block is always kept,
 *     with a causal mask inside it; the gate score is the inner product of
 *     the query with the mean-pooled keys.
 *   "When a MoBA reproduction will not run" (mhpq.cn/news/582794) section 3.3:
 *     attention over the selected blocks only.
 *
 * Selection rule (one rule, also used by the test oracle): query token i of a
 * sequence lies in block c_i = i / block_size.  It attends to block c_i (keys
 * up to and including i) and to the top (topk - 1) blocks among 0 .. c_i - 1
 * by the score <q_i, mean of the block's keys>, ties going to the lower block
 * index; when c_i <= topk - 1 it attends to every block 0 .. c_i.  Attention
 * is softmax(q k^T / sqrt(D)) v over those keys.  topk >= number of blocks
 * gives ordinary causal attention.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA
 *     memory) unless stated; the caller owns them.  Nothing is retained after
 *     the call returns.
 *   - q, k, v, out are bf16, laid out [B][S][H][D] (fixed length) or
 *     [total_tokens][H][D] (varlen, sequences packed back to back), dense and
 *     16-byte aligned.  D must be 64 or 128; H >= 1.
 *   - lse is fp32, natural log of the softmax denominator of the scaled
 *     logits: [B][H][S] (fixed length) or [H][total_tokens] (varlen).
 *   - block_size must be a positive multiple of 64; topk >= 1.  topk larger
 *     than the number of blocks is not an error (all blocks are kept).
 *     topk - 1 must be <= 31 unless topk covers every block.
 *   - total tokens (B * S) must be below 2^26.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  All work is
 *     enqueued on it; no entry point synchronises the host except
 *     moba_get_status.
 *   - Return value: MOBA_OK, or an error code.  Argument errors are detected
 *     on the host before anything is launched.  MOBA_ERR_CUDA reports a
 *     failed launch or allocation.  A kernel that gives up a bounded wait
 *     records MOBA_ERR_TIMEOUT in a device-side status word that
 *     moba_get_status reads.
 *   - Per-device state (that status word, the scratch of the allocation-free
 *     forward, the SM count) is allocated on first use and cached for the
 *     process, thread-safely.  cudaDeviceReset frees it behind the library's
 *     back: a process that resets a device must not call the library on that
 *     device again.
 */
#ifndef MOBA_GB300_H
#define MOBA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOBA_OK = 0,
    MOBA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad block_size/topk */
    MOBA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (D not 64/128, sizes too large) */
    MOBA_ERR_CUDA = 3,         /* a CUDA launch / allocation failed */
    MOBA_ERR_WORKSPACE = 4,    /* caller workspace too small */
    MOBA_ERR_TIMEOUT = 5       /* a kernel gave up a bounded wait (device status word) */
} moba_status_t;

/*
 * Per-call options of the _ex entry points.  Passing NULL, or a structure
 * whose fields are all zero, selects the defaults.  The library keeps no
 * process-wide setting: two threads may call with different options on
 * different streams at the same time.
 *
 *   pooling      how each block's keys are pooled into the representative the
 *                gate scores: MOBA_POOL_MEAN (default) = their mean ("Moonshot
 *                MoBA paper explained" section 3.1 mean_pool; "MOBA mixture of
 *                block attention for server-side long context" section 3);
 *                MOBA_POOL_MAX = their element-wise maximum, the variant the
 *                latter page also allows.
 *   gate_kernel  MOBA_GATE_TENSOR_CORES (default): block scores on the tensor
 *                cores (q times the pooled keys split into two bf16 terms,
 *                fp32 accumulation) and an exact fp32 re-score of the blocks
 *                inside a proven error margin of the top-(k-1) boundary; used
 *                while the longest sequence has at most 256 blocks, the CUDA
 *                cores above that.  MOBA_GATE_CUDA_CORES: every score on the
 *                CUDA cores.  Both select exactly the same blocks.
 *   attn_kernel  MOBA_ATTN_TCGEN05 (default): tcgen05 MMAs with TMEM
 *                accumulators and TMA-staged K/V; MOBA_ATTN_MMA_SYNC: the
 *                warp-level mma.sync kernels kept as the measured baseline.
 *                Same selection; results within the stated tolerances.
 *   debug_flags  test hook of the bounded waits: bit 0 makes the tcgen05
 *                attention's K/V producer skip its first load, so that the
 *                consumer's wait runs out and MOBA_ERR_TIMEOUT is recorded in
 *                the device status word instead of the GPU hanging.  0 in use.
 *   wait_limit_cycles  clock64 budget of one bounded wait; <= 0 keeps the
 *                default (about 2 s).
 *   idx_out      forward only, optional DEVICE int32 [tokens][H][topk]: the
 *                selection the call used (as moba_gate_topk writes it: the
 *                selected blocks ascending, -1 padded), written also on the
 *                paths that run no gate (top-1, and top-k covering every
 *                block).  4-byte aligned.
 *   schedule     forward only: MOBA_SCHEDULE_ADAPTIVE (default) lets a
 *                256-row job of one block and head whose rows together selected
 *                at most topk - 1 distinct past blocks attend to them in the
 *                own-block pass (query-major, each row masked to its own
 *                selection, no partial outputs; block sizes that are multiples
 *                of 256, topk <= 9, tcgen05 attention); every other row goes
 *                through the per-block lists.  MOBA_SCHEDULE_BLOCK_MAJOR sends
 *                every row through the lists.  Same results either way (within
 *                the stated tolerances).
 *   phase_events forward only, optional: an array of 7 cudaEvent_t (passed as
 *                void *) owned by the caller; the call records event i on its
 *                stream before phase i and event 6 after the last one.  Phases:
 *                0 sequence tables, 1 key pooling, 2 gate + top-k, 3 regroup,
 *                4 attention over past blocks, 5 attention over the own block
 *                + merge (a phase a path skips is empty).  A NULL entry is
 *                skipped.
 *   idx_in       backward only, optional DEVICE int32 [tokens][H][topk]: the
 *                selection of the forward pass (its idx_out), saved by the
 *                caller like lse.  The backward then regroups this selection
 *                instead of recomputing it (no key pooling, no gate).  A row's
 *                past blocks are read in order up to the first entry that is
 *                negative or not below the row's own block; values are not
 *                otherwise checked (a different selection gives the gradients
 *                of that selection).  4-byte aligned.  NULL: recompute.
 * An option value outside its set returns MOBA_ERR_INVALID_ARG before any
 * launch.
 */
enum { MOBA_POOL_MEAN = 0, MOBA_POOL_MAX = 1 };
enum { MOBA_GATE_TENSOR_CORES = 0, MOBA_GATE_CUDA_CORES = 1 };
enum { MOBA_ATTN_TCGEN05 = 0, MOBA_ATTN_MMA_SYNC = 1 };
enum { MOBA_SCHEDULE_ADAPTIVE = 0, MOBA_SCHEDULE_BLOCK_MAJOR = 1 };
enum { MOBA_NUM_PHASES = 6 };

typedef struct moba_options {
    int pooling;
    int gate_kernel;
    int attn_kernel;
    int debug_flags;
    long long wait_limit_cycles;
    int32_t *idx_out;
    void *const *phase_events;
    int schedule;
    const int32_t *idx_in;
} moba_options_t;

/* Number of blocks of a sequence: ceil(len / block_size) (the tail block may
 * be partial).  "Moonshot MoBA paper explained" section 4.1 divides the
 * context length by the block size (32768 / 512 = 64). */
int moba_num_blocks(int len, int block_size);

/*
 * Mean-pooled keys ("Moonshot MoBA paper explained" section 3.1, mean_pool).
 *   k    : [B][S][H][D] bf16 (device)
 *   kbar : [B * n][H][D] fp32 (device, written), n = moba_num_blocks(S, bs);
 *          kbar[b*n + c][h][:] = mean of k[b][t][h][:] over the tokens t of
 *          block c (the tail block averages only the tokens it holds).
 *          Blocks are the outer index (not heads) so that the pooled keys of
 *          packed variable-length sequences concatenate like their tokens do.
 * moba_kpool_ex takes the per-call options (only `pooling` applies).
 */
int moba_kpool(const void *k, float *kbar, int B, int H, int S, int D, int block_size,
               void *stream);
int moba_kpool_ex(const void *k, float *kbar, int B, int H, int S, int D, int block_size,
                  const moba_options_t *options, void *stream);

/* Varlen form: k [total_tokens][H][D]; cu_seqlens is a DEVICE int32 array of
 * num_seqs + 1 prefix offsets (cu_seqlens[num_seqs] == total_tokens).
 * kbar: [sum over sequences of n_b][H][D], sequence 0's blocks first. */
int moba_kpool_varlen(const void *k, float *kbar, const int32_t *cu_seqlens, int num_seqs,
                      int total_tokens, int H, int D, int block_size, void *stream);
int moba_kpool_varlen_ex(const void *k, float *kbar, const int32_t *cu_seqlens, int num_seqs,
                         int total_tokens, int H, int D, int block_size,
                         const moba_options_t *options, void *stream);

/*
 * Gate and top-k selection ("Moonshot MoBA paper explained" sections 3.1 and
 * 4.1; "MOBA ... server-side long context" section 3).  Scores are
 * <q, kbar> in fp32 for the strictly-past blocks only.
 *   q    : [B][S][H][D] bf16 (device)
 *   kbar : as written by moba_kpool (device)
 *   idx  : [B][S][H][topk] int32 (device, written): the selected local block
 *          ids of each (token, head) in ascending order (the own block is
 *          therefore last among the valid entries), padded with -1.
 */
int moba_gate_topk(const void *q, const float *kbar, int32_t *idx, int B, int H, int S, int D,
                   int block_size, int topk, void *stream);
/* with per-call options (only `gate_kernel` applies) */
int moba_gate_topk_ex(const void *q, const float *kbar, int32_t *idx, int B, int H, int S, int D,
                      int block_size, int topk, const moba_options_t *options, void *stream);

/* Varlen form of moba_gate_topk: q [total_tokens][H][D], idx
 * [total_tokens][H][topk]; cu_seqlens as for moba_kpool_varlen. */
int moba_gate_topk_varlen(const void *q, const float *kbar, int32_t *idx,
                          const int32_t *cu_seqlens, int num_seqs, int total_tokens, int H,
                          int D, int block_size, int topk, void *stream);
int moba_gate_topk_varlen_ex(const void *q, const float *kbar, int32_t *idx,
                             const int32_t *cu_seqlens, int num_seqs, int total_tokens, int H,
                             int D, int block_size, int topk, const moba_options_t *options,
                             void *stream);

/*
 * Full MoBA forward: pool, gate, regroup of the queries by selected block,
 * attention over the past blocks, causal attention inside the own block and
 * the log-sum-exp merge of the partial results.
 *   q, k, v : [B][S][H][D] bf16 (device);  out : [B][S][H][D] bf16 (device)
 *   lse     : [B][H][S] fp32 (device)
 * Scratch is allocated stream-ordered on `stream` (cudaMallocAsync) and
 * released on the same stream before returning.
 */
int moba_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                  int H, int S, int D, int block_size, int topk, void *stream);

/* Bytes of device scratch moba_attn_fwd_ws / _ex need for these sizes (the
 * same for every option); moba_workspace_size is the same function. */
size_t moba_attn_fwd_workspace_size(int B, int H, int S, int D, int block_size, int topk);
size_t moba_workspace_size(int B, int H, int S, int D, int block_size, int topk);

/* moba_attn_fwd with caller-provided device scratch (256-byte aligned,
 * at least moba_attn_fwd_workspace_size bytes; MOBA_ERR_WORKSPACE if
 * smaller).  The scratch must not be used by anything else until the work
 * enqueued on `stream` has finished. */
int moba_attn_fwd_ws(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int H, int S, int D, int block_size, int topk, void *workspace,
                     size_t workspace_bytes, void *stream);

/* moba_attn_fwd with per-call options (NULL = defaults).  workspace may be
 * NULL (scratch from cudaMallocAsync on the stream, as moba_attn_fwd) or the
 * caller's scratch (as moba_attn_fwd_ws). */
int moba_attn_fwd_ex(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                     int H, int S, int D, int block_size, int topk, const moba_options_t *options,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * moba_attn_fwd on HOST buffers: the same operation and layouts, with q, k,
 * v, out and lse in host memory (page-locked for asynchronous copies; other
 * host memory works but the copies then block).  Enqueued on `stream` and
 * returning before completion: k, q and v are copied to the device scratch in
 * that order on a stream of the call's own, starting after the earlier work
 * on `stream`; the pooling, the gate
 * and the attention each wait only for the inputs they read, so the first
 * phases run while v is still arriving; out and lse come back the same way,
 * and `stream` reaches its next work once they have.  The host buffers must
 * stay valid, and out / lse unread, until then.  Two calls on different
 * streams with different scratch run side by side (one call's copies beside
 * the other's kernels).
 *   dev_scratch : device memory, 256-byte aligned, at least
 *                 moba_attn_fwd_host_scratch_size bytes (MOBA_ERR_WORKSPACE
 *                 otherwise): the device copies of q, k, v, out, lse and the
 *                 forward's workspace; not used by anything else until the
 *                 call's work has finished.
 *   options     : as moba_attn_fwd_ex (idx_out, if given, is device memory).
 * Errors: as moba_attn_fwd_ex; a failed copy or stream/event creation
 * returns MOBA_ERR_CUDA.
 */
int moba_attn_fwd_host(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                       int H, int S, int D, int block_size, int topk,
                       const moba_options_t *options, void *dev_scratch, size_t scratch_bytes,
                       void *stream);
size_t moba_attn_fwd_host_scratch_size(int B, int H, int S, int D, int block_size, int topk);

/*
 * Varlen forward: q, k, v, out [total_tokens][H][D] bf16; lse
 * [H][total_tokens] fp32; cu_seqlens DEVICE int32 [num_seqs + 1];
 * max_seqlen >= every sequence length.  Each sequence is partitioned into
 * its own blocks starting at its first token.
 * cu_seqlens lives on the device, so its consistency is checked there, by the
 * first kernel of the call: it must start at 0, never decrease, give no
 * sequence more than max_seqlen tokens and end at total_tokens.  When it does
 * not, no later kernel of the call reads or writes anything through it, out
 * and lse are left unwritten, and MOBA_ERR_INVALID_ARG is recorded in the
 * device status word (read it with moba_get_status).  The same check guards
 * every varlen entry point.
 */
int moba_attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                         const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                         int max_seqlen, int H, int D, int block_size, int topk, void *stream);

size_t moba_attn_fwd_varlen_workspace_size(int num_seqs, int total_tokens, int max_seqlen, int H,
                                           int D, int block_size, int topk);

int moba_attn_fwd_varlen_ex(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                            int max_seqlen, int H, int D, int block_size, int topk,
                            const moba_options_t *options, void *workspace,
                            size_t workspace_bytes, void *stream);

int moba_attn_fwd_varlen_ws(const void *q, const void *k, const void *v, void *out, float *lse,
                            const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                            int max_seqlen, int H, int D, int block_size, int topk,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass of moba_attn_fwd: the gradients of the MoBA attention with
 * the gate's selection held fixed (top-k is piecewise constant and passes no
 * gradient; none reaches the pooled keys).  "MOBA ... server-side long
 * context" section 3 trains MoBA layers end to end; the selection is the
 * forward's ("Moonshot MoBA paper explained" sections 3.1 and 4.1), recomputed
 * here with the same kernels.
 *   q, k, v   : [B][S][H][D] bf16 (device), the forward's inputs
 *   out, lse  : the forward's results ([B][S][H][D] bf16, [B][H][S] fp32)
 *   dout      : [B][S][H][D] bf16 (device), dL/d(out)
 *   dq, dk, dv: [B][S][H][D] bf16 (device, written)
 * The summation order follows the GPU's scheduling (the per-block query lists
 * fill in any order; dq adds fp32 atomics), so results may differ between
 * calls in their last bits.
 * Host-side argument errors (null or 16-byte-misaligned tensors, the sizes
 * moba_attn_fwd rejects) return before any launch.  Scratch (the forward's
 * selection tables and lists, an fp32 dq accumulator of B*S*H*D floats and
 * B*S*H floats of dO . O) comes from cudaMallocAsync on `stream`; the _ws form
 * takes it from the caller (256-byte aligned, at least
 * moba_attn_bwd_workspace_size bytes, else MOBA_ERR_WORKSPACE).
 */
int moba_attn_bwd(const void *q, const void *k, const void *v, const void *out,
                  const float *lse, const void *dout, void *dq, void *dk, void *dv, int B, int H,
                  int S, int D, int block_size, int topk, void *stream);
size_t moba_attn_bwd_workspace_size(int B, int H, int S, int D, int block_size, int topk);
int moba_attn_bwd_ws(const void *q, const void *k, const void *v, const void *out,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                     int H, int S, int D, int block_size, int topk, void *workspace,
                     size_t workspace_bytes, void *stream);
/* with per-call options (pooling and gate_kernel decide the recomputed
 * selection and must match the forward's); workspace may be NULL */
int moba_attn_bwd_ex(const void *q, const void *k, const void *v, const void *out,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                     int H, int S, int D, int block_size, int topk, const moba_options_t *options,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Varlen backward: every tensor [total_tokens][H][D] bf16, lse [H][total_tokens]
 * fp32 as moba_attn_fwd_varlen wrote it; cu_seqlens DEVICE int32. */
int moba_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *out,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                         int max_seqlen, int H, int D, int block_size, int topk, void *stream);
size_t moba_attn_bwd_varlen_workspace_size(int num_seqs, int total_tokens, int max_seqlen, int H,
                                           int D, int block_size, int topk);
int moba_attn_bwd_varlen_ex(const void *q, const void *k, const void *v, const void *out,
                            const float *lse, const void *dout, void *dq, void *dk, void *dv,
                            const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                            int max_seqlen, int H, int D, int block_size, int topk,
                            const moba_options_t *options, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * moba_attn_fwd for callers that cannot allocate device memory: for example
 * code running under a memory manager that owns the whole device (where an
 * extra cudaMalloc can fail or fragment its pool), or a serving loop that must
 * not allocate on its latency path.  The pages describe no such entry point;
 * it is an addition of this library.
 *   Arguments, layouts and results are those of moba_attn_fwd; the caller
 *   still passes q, k, v, out and lse.
 *   Scratch: one file-scope device array of moba_attn_fwd_noalloc_capacity()
 *   bytes (64 MiB), held by every device that loads this library until the
 *   process exits.  Sizes whose scratch (moba_attn_fwd_workspace_size) does not
 *   fit return MOBA_ERR_WORKSPACE before anything is launched.
 *   No cudaMalloc, cudaFree or allocating library routine is called.  The
 *   first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.
 *   Every call shares the one array and it keeps the previous call's contents
 *   (what must start at zero is cleared by the call): calls whose work
 *   overlaps on the GPU, e.g. on two streams, race and must be serialised by
 *   the caller.
 */
int moba_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int S, int D, int block_size, int topk, void *stream);

/* Bytes of the static scratch array used by moba_attn_fwd_noalloc. */
size_t moba_attn_fwd_noalloc_capacity(void);

/* Synchronises `stream`, returns the device status word of the current device
 * (MOBA_OK, MOBA_ERR_TIMEOUT from a bounded wait, or MOBA_ERR_INVALID_ARG from
 * inconsistent device-side lengths) and clears it; MOBA_ERR_CUDA if the
 * synchronisation itself failed.  The word is per device, shared by all
 * streams: a call reports what any earlier work on the device recorded. */
int moba_get_status(void *stream);

/* Static, human-readable name of a status code. */
const char *moba_status_string(int code);

/* Text of the CUDA error behind the calling thread's last MOBA_ERR_CUDA
 * ("no error" if there was none). */
const char *moba_last_cuda_error(void);

/* Number of kernels this library has launched since it was loaded (a
 * process-wide tally, counted atomically; host only). */
unsigned long long moba_launch_count(void);

/*
 * Decode: one new query token per sequence against its KV cache.  The step
 * computes exactly what the prefill forward computes for the sequence's last
 * row i = len - 1 ("Moonshot MoBA paper explained" sections 3.1 and 4.1;
 * "MOBA mixture of block attention for server-side long context" section 3):
 * the top (topk - 1) past blocks by <q, kbar> plus the own block, softmax
 * attention over their keys (the own block up to i).  Selections equal those
 * of moba_gate_topk for that row.
 *   q          : [B][H][D] bf16 (device), the new token's queries
 *   k_cache,
 *   v_cache    : [B][S_max][H][D] bf16 (device); the new token's k and v are
 *                already written at position cache_lens[b] - 1
 *   kbar       : the pooled keys of the caches as written by moba_kpool over
 *                k_cache with S = S_max (fp32, [B * ceil(S_max/bs)][H][D]);
 *                only the blocks before each row's own block are read, so a
 *                caller may keep it current by pooling each block once it is
 *                complete
 *   cache_lens : [B] int32 (device), 1 <= len <= S_max; a length outside
 *                that range gives that sequence zero output and -inf lse and
 *                MOBA_ERR_INVALID_ARG in the device status word
 *   out        : [B][H][D] bf16 (device, written); lse: [B][H] fp32 (natural
 *                log, written); idx: [B][H][topk] int32 or NULL (the
 *                selection, ascending, -1 padded)
 * Host-side argument errors return before any launch; topk - 1 above 32
 * while topk is below ceil(S_max / bs) is MOBA_ERR_UNSUPPORTED.  The plain
 * form takes its scratch from cudaMallocAsync on the stream; the _ws form
 * takes it from the caller (256-byte aligned, at least
 * moba_decode_workspace_size bytes; it allocates nothing).
 */
int moba_decode_fwd(const void *q, const void *k_cache, const void *v_cache, const float *kbar,
                    const int32_t *cache_lens, void *out, float *lse, int32_t *idx, int B, int H,
                    int S_max, int D, int block_size, int topk, void *stream);
size_t moba_decode_workspace_size(int B, int H, int D, int topk);
int moba_decode_fwd_ws(const void *q, const void *k_cache, const void *v_cache,
                       const float *kbar, const int32_t *cache_lens, void *out, float *lse,
                       int32_t *idx, int B, int H, int S_max, int D, int block_size, int topk,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Where the timeout reported by the calling thread's last moba_get_status
 * happened: out4 = {barrier shared-memory address, parity, block index, thread
 * index}. */
void moba_debug_timeout_info(int *out4);

#ifdef __cplusplus
}
#endif

#endif /* MOBA_GB300_H */
