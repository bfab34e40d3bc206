/*
 * moba_oracle.c -- plain, slow CPU oracle of the Mixture of Block Attention
 * (MoBA) forward and backward passes.  TEST INFRASTRUCTURE ONLY: the tests,
 * the smoke check and the CPU-baseline leg of the benchmark call it; the CUDA
 * library never does, and the two share no code.
 *
 * Pages this follows (cited by page title and section):
 *   [P2] "Moonshot MoBA paper explained: sparse-attention config skeleton"
 *        (gsyq.cn/news/227272), sections 1, 3.1, 4.1, 5.
 *   [P4] "MOBA mixture of block attention for server-side long context"
 *        (hncyxsy.com/news/197418), sections 1, 3.
 *   [P1] "When a MoBA reproduction will not run" (mhpq.cn/news/582794),
 *        sections 1.2, 3.1-3.3 (questions about the method's edge cases).
 *
 * Everything is accumulated in double precision.  Inputs are the bf16 bit
 * patterns of q, k, v, widened exactly to double.
 *
 * Layouts (all row-major, "token-major" like FlashAttention's varlen API):
 *   q, k, v   : [total_tokens][H][D] bf16 bits (uint16)
 *   cu_seqlens: [num_seqs + 1] int64 prefix offsets of the packed sequences
 *   kbar      : [num_blocks_total][H][D] double, blocks of sequence b first
 *   rows      : (global token, head) pairs whose outputs are wanted
 *
 * Readings where the pages are silent (each is stated where it is used):
 *   R1 block count is ceil(len / block_size); the tail block may be partial.
 *   R2 gate score is the raw inner product q . kbar (no scale, no softmax:
 *      both are monotone and cannot change the selected set).
 *   R3 the query's own block is always selected and counts toward top-k;
 *      the other k-1 are the highest-scoring strictly-past blocks; ties go to
 *      the lower block index; with fewer than k-1 past blocks all are kept.
 *   R4 attention logits are scaled by 1/sqrt(D); lse is the natural log of
 *      the softmax denominator of the scaled logits.
 *   R5 gating is per (sequence, head): each head pools its own keys.
 *   R6 max pooling (the variant the server-side page allows) takes the
 *      element-wise maximum over the block's own tokens.
 *   R7 the backward pass holds the gate's selection fixed (top-k is piecewise
 *      constant, so it passes no gradient; none reaches the pooled keys):
 *      gradients flow through the softmax attention over the selected keys
 *      only.  [P4] section 3 trains MoBA layers end to end (it blames the
 *      sparse gradient path for a higher SFT loss).
 *
 * Parity pins for every function here live in tests/test_oracle.py (forward)
 * and tests/test_oracle_bwd.py (backward).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* R1 -- [P2] section 4.1 computes the block count of a 32768-token context
 * with block size 512 as 64; [P1] section 3.1 asks what happens when the
 * length is not a multiple of the block size.  Reading: round up, so the
 * last block holds the remainder. */
int64_t moba_oracle_num_blocks(int64_t len, int64_t block_size)
{
    if (len <= 0 || block_size <= 0) return 0;
    return (len + block_size - 1) / block_size;
}

int moba_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Global index of the first block of every sequence ([num_seqs + 1]). */
static int64_t *block_bases(const int64_t *cu, int num_seqs, int64_t bs)
{
    int64_t *base = (int64_t *)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
    if (!base) return NULL;
    base[0] = 0;
    for (int b = 0; b < num_seqs; ++b)
        base[b + 1] = base[b] + moba_oracle_num_blocks(cu[b + 1] - cu[b], bs);
    return base;
}

/* Step "block representation" -- [P2] section 3.1 (score_fn = mean_pool:
 * average the keys inside the block) and [P4] section 3 (the gate uses the
 * keys mean-pooled along the sequence).  kbar[g][h][d] = mean over the
 * tokens t of block g of k[t][h][d]. */
int moba_oracle_kpool(const uint16_t *k, const int64_t *cu, int num_seqs,
                      int H, int D, int block_size, double *kbar)
{
    if (!k || !cu || !kbar || num_seqs < 1 || H < 1 || D < 1 || block_size < 1)
        return -1;
    int64_t *base = block_bases(cu, num_seqs, block_size);
    if (!base) return -2;
    const int64_t HD = (int64_t)H * D;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t t_begin = cu[b], len = cu[b + 1] - cu[b];
        int64_t n = base[b + 1] - base[b];
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t c = 0; c < n; ++c) {
            int64_t g = base[b] + c;
            int64_t t0 = t_begin + c * block_size;
            int64_t t1 = t0 + block_size;
            if (t1 > t_begin + len) t1 = t_begin + len;
            double *sum = kbar + g * HD;
            for (int64_t e = 0; e < HD; ++e) sum[e] = 0.0;
            /* every element sums its block's tokens in ascending order */
            for (int64_t t = t0; t < t1; ++t) {
                const uint16_t *row = k + t * HD;
                for (int64_t e = 0; e < HD; ++e) sum[e] += widen_bf16(row[e]);
            }
            for (int64_t e = 0; e < HD; ++e) sum[e] /= (double)(t1 - t0);
        }
    }
    free(base);
    return 0;
}

/*
 * Max-pooled keys: kbar[g][h][d] = max over the tokens t of block g of
 * k[t][h][d] ([P4] section 3 allows max pooling along the sequence instead of
 * the mean: it reacts more to blocks dense in key information).  Reading R6:
 * the maximum is taken per element (per head and dimension), over the block's
 * own tokens only (a partial tail block included).  Exact in any precision.
 */
int moba_oracle_kpool_max(const uint16_t *k, const int64_t *cu, int num_seqs,
                          int H, int D, int block_size, double *kbar)
{
    if (!k || !cu || !kbar || num_seqs < 1 || H < 1 || D < 1 || block_size < 1)
        return -1;
    int64_t *base = block_bases(cu, num_seqs, block_size);
    if (!base) return -2;
    const int64_t HD = (int64_t)H * D;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t t_begin = cu[b], len = cu[b + 1] - cu[b];
        int64_t n = base[b + 1] - base[b];
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t c = 0; c < n; ++c) {
            int64_t g = base[b] + c;
            int64_t t0 = t_begin + c * block_size;
            int64_t t1 = t0 + block_size;
            if (t1 > t_begin + len) t1 = t_begin + len;
            double *mx = kbar + g * HD;
            for (int64_t e = 0; e < HD; ++e) mx[e] = widen_bf16(k[t0 * HD + e]);
            for (int64_t t = t0 + 1; t < t1; ++t) {
                const uint16_t *row = k + t * HD;
                for (int64_t e = 0; e < HD; ++e) {
                    const double x = widen_bf16(row[e]);
                    if (x > mx[e]) mx[e] = x;
                }
            }
        }
    }
    free(base);
    return 0;
}

typedef struct {
    double score;
    int64_t block;
} candidate_t;

/* Order used by top-k: higher score first; equal scores -> lower block. */
static int by_score_then_block(const void *pa, const void *pb)
{
    const candidate_t *a = (const candidate_t *)pa, *b = (const candidate_t *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->block < b->block) ? -1 : (a->block > b->block);
}

static int by_block(const void *pa, const void *pb)
{
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    return (a < b) ? -1 : (a > b);
}

/*
 * Forward pass for a list of rows.
 *
 * For each row r (token t = row_tok[r], head h = row_head[r]):
 *  gate   -- [P2] 3.1 (mean-pool affinity, future blocks masked),
 *            [P2] 4.1 (sort all block scores, keep the top_k),
 *            [P4] 3 (force_current_block: the own block always attends with a
 *            causal mask inside it); readings R2, R3, R5.
 *            Block c of the row's sequence is scored only if c < c_i, the
 *            row's own block; the current block is never scored (its mean
 *            would include future keys).
 *  attend -- softmax attention over the keys of the selected blocks that are
 *            not after the query ([P1] 3.3: selected blocks go to
 *            FlashAttention with a causal mask inside the current block;
 *            unselected blocks contribute nothing, reading of [P1] 3.2's
 *            question); reading R4.
 *
 * Outputs per row: idx[r][0..topk) -- selected local block ids ascending,
 * -1 padded; gap[r] -- score of the last past block kept minus the best past
 * block dropped (INFINITY when nothing had to be dropped); o[r][0..D) and
 * lse[r].  If given_idx is not NULL the gate is skipped and its rows are used
 * as the selection (entries < 0 ignored); gap is then INFINITY.
 */
int moba_oracle_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int64_t *cu, int num_seqs, int H, int D,
                     int block_size, int topk, const double *kbar,
                     int64_t nrows, const int64_t *row_tok,
                     const int32_t *row_head, const int32_t *given_idx,
                     int32_t *idx_out, double *gap_out, double *o_out,
                     double *lse_out)
{
    if (!q || !k || !v || !cu || !kbar || !row_tok || !row_head || !idx_out ||
        !gap_out || !o_out || !lse_out)
        return -1;
    if (num_seqs < 1 || H < 1 || D < 1 || block_size < 1 || topk < 1)
        return -1;
    int64_t *base = block_bases(cu, num_seqs, block_size);
    if (!base) return -2;
    const double scale = 1.0 / sqrt((double)D);
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = row_tok[r];
        int h = row_head[r];
        /* sequence that holds token t */
        int lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        int b = lo;
        int64_t t_begin = cu[b], len = cu[b + 1] - cu[b];
        if (t < t_begin || t >= t_begin + len || h < 0 || h >= H) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        int64_t i = t - t_begin;            /* position inside the sequence */
        int64_t ci = i / block_size;        /* the row's own block */
        int64_t n = moba_oracle_num_blocks(len, block_size);

        /* ---------------- gate ---------------- */
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n + 1));
        int64_t nsel = 0;
        double gap = INFINITY;
        if (given_idx) {
            for (int j = 0; j < topk; ++j) {
                int32_t c = given_idx[r * topk + j];
                if (c >= 0 && c <= ci) sel[nsel++] = c;
            }
        } else {
            int64_t keep_past = (int64_t)topk - 1;
            if (ci <= keep_past) {
                /* fewer past blocks than slots: keep them all */
                for (int64_t c = 0; c < ci; ++c) sel[nsel++] = c;
            } else if (keep_past > 0) {
                candidate_t *cand =
                    (candidate_t *)malloc(sizeof(candidate_t) * (size_t)ci);
                const uint16_t *qrow = q + (t * H + h) * D;
                for (int64_t c = 0; c < ci; ++c) {
                    const double *kb = kbar + ((base[b] + c) * H + h) * D;
                    double s = 0.0;
                    for (int d = 0; d < D; ++d) s += widen_bf16(qrow[d]) * kb[d];
                    cand[c].score = s;
                    cand[c].block = c;
                }
                qsort(cand, (size_t)ci, sizeof(candidate_t), by_score_then_block);
                for (int64_t j = 0; j < keep_past; ++j) sel[nsel++] = cand[j].block;
                gap = cand[keep_past - 1].score - cand[keep_past].score;
                free(cand);
            }
            sel[nsel++] = ci; /* forced current block */
        }
        qsort(sel, (size_t)nsel, sizeof(int64_t), by_block);
        for (int j = 0; j < topk; ++j)
            idx_out[r * topk + j] = (j < nsel) ? (int32_t)sel[j] : -1;
        gap_out[r] = gap;

        /* ---------------- attend ---------------- */
        int64_t nkeys = 0;
        for (int64_t j = 0; j < nsel; ++j) {
            int64_t k0 = sel[j] * block_size, k1 = k0 + block_size;
            if (k1 > i + 1) k1 = i + 1; /* causal: keys at or before the query */
            if (k1 > k0) nkeys += k1 - k0;
        }
        double *z = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
        int64_t *kt = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nkeys > 0 ? nkeys : 1));
        const uint16_t *qrow = q + (t * H + h) * D;
        int64_t m_idx = 0;
        for (int64_t j = 0; j < nsel; ++j) {
            int64_t k0 = sel[j] * block_size, k1 = k0 + block_size;
            if (k1 > i + 1) k1 = i + 1;
            for (int64_t p = k0; p < k1; ++p) {
                const uint16_t *krow = k + ((t_begin + p) * H + h) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += widen_bf16(qrow[d]) * widen_bf16(krow[d]);
                z[m_idx] = dot * scale;
                kt[m_idx] = t_begin + p;
                ++m_idx;
            }
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) if (z[j] > m) m = z[j];
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) l += exp(z[j] - m);
        double *orow = o_out + r * D;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            double w = exp(z[j] - m) / l;
            const uint16_t *vrow = v + (kt[j] * H + h) * D;
            for (int d = 0; d < D; ++d) orow[d] += w * widen_bf16(vrow[d]);
        }
        lse_out[r] = m + log(l);
        free(z);
        free(kt);
        free(sel);
    }
    free(base);
    return failed ? -3 : 0;
}

/*
 * Backward pass of one row (reading R7): the softmax attention of row i of
 * sequence b, head h over the keys of its selected blocks, differentiated.
 * With z_j = (q . k_j) / sqrt(D), P_j = exp(z_j - lse), o = sum_j P_j v_j and
 * the upstream gradient g = dL/do:
 *   dP_j = g . v_j,  delta = g . o,  dz_j = P_j (dP_j - delta)
 *   dL/dq   = sum_j dz_j k_j / sqrt(D)
 *   dL/dk_j += dz_j q / sqrt(D),   dL/dv_j += P_j g
 * dq_row receives dL/dq; dk, dv (whole [total][H][D] arrays) are accumulated
 * into when not NULL.  sel holds the nsel selected local blocks.
 */
static void row_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int64_t t_begin, int64_t i, int h,
                         int H, int D, int block_size, const int64_t *sel,
                         int64_t nsel, double *dq_row, double *dk, double *dv)
{
    const double scale = 1.0 / sqrt((double)D);
    const int64_t t = t_begin + i;
    int64_t nkeys = 0;
    for (int64_t j = 0; j < nsel; ++j) {
        int64_t k0 = sel[j] * block_size, k1 = k0 + block_size;
        if (k1 > i + 1) k1 = i + 1;
        if (k1 > k0) nkeys += k1 - k0;
    }
    double *z = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
    int64_t *kt = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nkeys > 0 ? nkeys : 1));
    double *o = (double *)calloc((size_t)D, sizeof(double));
    const uint16_t *qrow = q + (t * H + h) * D;
    const uint16_t *grow = dout + (t * H + h) * D;
    int64_t n = 0;
    for (int64_t j = 0; j < nsel; ++j) {
        int64_t k0 = sel[j] * block_size, k1 = k0 + block_size;
        if (k1 > i + 1) k1 = i + 1;
        for (int64_t p = k0; p < k1; ++p) {
            const uint16_t *krow = k + ((t_begin + p) * H + h) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += widen_bf16(qrow[d]) * widen_bf16(krow[d]);
            z[n] = dot * scale;
            kt[n] = t_begin + p;
            ++n;
        }
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) if (z[j] > m) m = z[j];
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) l += exp(z[j] - m);
    /* z now holds P_j */
    for (int64_t j = 0; j < nkeys; ++j) z[j] = exp(z[j] - m) / l;
    for (int64_t j = 0; j < nkeys; ++j) {
        const uint16_t *vrow = v + (kt[j] * H + h) * D;
        for (int d = 0; d < D; ++d) o[d] += z[j] * widen_bf16(vrow[d]);
    }
    double delta = 0.0;
    for (int d = 0; d < D; ++d) delta += widen_bf16(grow[d]) * o[d];
    for (int d = 0; d < D; ++d) dq_row[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const uint16_t *krow = k + (kt[j] * H + h) * D;
        const uint16_t *vrow = v + (kt[j] * H + h) * D;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += widen_bf16(grow[d]) * widen_bf16(vrow[d]);
        const double dz = z[j] * (dp - delta);
        for (int d = 0; d < D; ++d) dq_row[d] += dz * widen_bf16(krow[d]) * scale;
        if (dk) {
            double *dkr = dk + (kt[j] * H + h) * D;
            for (int d = 0; d < D; ++d) dkr[d] += dz * widen_bf16(qrow[d]) * scale;
        }
        if (dv) {
            double *dvr = dv + (kt[j] * H + h) * D;
            for (int d = 0; d < D; ++d) dvr[d] += z[j] * widen_bf16(grow[d]);
        }
    }
    free(o);
    free(kt);
    free(z);
}

/* The selected local blocks of one row, from a [.][topk] selection table
 * (entries < 0 or after the row's own block ignored). */
static int64_t row_selection(const int32_t *idx_row, int topk, int64_t ci, int64_t *sel)
{
    int64_t nsel = 0;
    for (int j = 0; j < topk; ++j) {
        int32_t c = idx_row[j];
        if (c >= 0 && c <= ci) sel[nsel++] = c;
    }
    return nsel;
}

/*
 * Gradients dq, dk, dv ([total][H][D], double) of the MoBA attention for the
 * upstream gradient dout ([total][H][D] bf16 bits), with the selection idx
 * ([total][H][topk], as the forward's gate returns it) held fixed.  Each
 * (sequence, head) pair is independent; its rows run in order.
 */
int moba_oracle_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const uint16_t *dout, const int64_t *cu, int num_seqs, int H, int D,
                    int block_size, int topk, const int32_t *idx, double *dq,
                    double *dk, double *dv)
{
    if (!q || !k || !v || !dout || !cu || !idx || !dq || !dk || !dv) return -1;
    if (num_seqs < 1 || H < 1 || D < 1 || block_size < 1 || topk < 1) return -1;
    const int64_t total = cu[num_seqs];
    memset(dk, 0, sizeof(double) * (size_t)(total * H * D));
    memset(dv, 0, sizeof(double) * (size_t)(total * H * D));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)num_seqs * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        const int64_t t_begin = cu[b], len = cu[b + 1] - cu[b];
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)topk);
        for (int64_t i = 0; i < len; ++i) {
            const int64_t t = t_begin + i;
            const int64_t nsel = row_selection(idx + (t * H + h) * topk, topk,
                                               i / block_size, sel);
            row_backward(q, k, v, dout, t_begin, i, h, H, D, block_size, sel, nsel,
                         dq + (t * H + h) * D, dk, dv);
        }
        free(sel);
    }
    return 0;
}

/* dq alone for a list of (token, head) rows -- the part of the backward that
 * a single row determines, for sampled checks at sizes the whole pass would
 * take too long on.  idx holds the listed rows' selections ([nrows][topk]). */
int moba_oracle_bwd_dq_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const uint16_t *dout, const int64_t *cu, int num_seqs, int H,
                            int D, int block_size, int topk, int64_t nrows,
                            const int64_t *row_tok, const int32_t *row_head,
                            const int32_t *idx, double *dq)
{
    if (!q || !k || !v || !dout || !cu || !row_tok || !row_head || !idx || !dq) return -1;
    if (num_seqs < 1 || H < 1 || D < 1 || block_size < 1 || topk < 1) return -1;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t t = row_tok[r];
        const int h = row_head[r];
        int lo = 0, hi = num_seqs - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        if (t < cu[lo] || t >= cu[lo + 1] || h < 0 || h >= H) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const int64_t i = t - cu[lo];
        int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)topk);
        const int64_t nsel = row_selection(idx + r * topk, topk, i / block_size, sel);
        row_backward(q, k, v, dout, cu[lo], i, h, H, D, block_size, sel, nsel, dq + r * D,
                     NULL, NULL);
        free(sel);
    }
    return failed ? -3 : 0;
}
