/*
 * oracle.c -- plain, slow CPU reference for split-KV attention forward.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
 * CPU-baseline leg are its only callers; the CUDA library never loads it and the
 * two share no code. Page citations use the tags defined in oracle.h:
 *   [P1] "Recombine fully masked split-KV attention partials on the host"
 *   [P2] "[ASM] [HIP] [JIT] [gfx942] Optimize long-context FMHA with split-KV"
 *
 * Pins (what checks this file against something other than itself) live in
 * tests/test_oracle_pins.py: the worked split counts printed on [P1], the review
 * notes' conservativeness bound checked by brute force, closed forms of
 * attention, a library attention routine in double precision, and the identity
 * that merging the partials gives unsplit attention.
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ inputs */

/* Exact conversion of one stored element to double. */
static double orc_load(orc_array a, int64_t idx)
{
    switch (a.dtype) {
    case ORC_BF16: {
        /* bfloat16 is the upper half of an IEEE binary32 word */
        uint32_t w = (uint32_t)((const uint16_t *)a.data)[idx] << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    case ORC_F16: {
        /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
        uint16_t h = ((const uint16_t *)a.data)[idx];
        int sign = (h >> 15) & 1;
        int e = (h >> 10) & 0x1f;
        int m = h & 0x3ff;
        double x;
        if (e == 0)
            x = ldexp((double)m, -24);                 /* zero or subnormal */
        else if (e == 31)
            x = (m == 0) ? INFINITY : NAN;
        else
            x = ldexp((double)(m + 1024), e - 25);     /* 1.m * 2^(e-15) */
        return sign ? -x : x;
    }
    case ORC_F32:
        return (double)((const float *)a.data)[idx];
    default:
        return ((const double *)a.data)[idx];
    }
}

int orc_check_problem(const orc_problem *p)
{
    if (!p || p->B < 0 || p->H <= 0 || p->d_qk <= 0 || p->d_v <= 0)
        return -1;
    if (!p->cu_q || !p->cu_k)
        return -1;
    if (p->n_per_block <= 0 || p->split_kv <= 0 || p->block_m <= 0)
        return -1;                                     /* [P1] assert(nPerBlock > 0) */
    if (p->mask < ORC_MASK_NONE || p->mask > ORC_MASK_PREFIX_CAUSAL)
        return -1;
    if (p->last_valid_kv_index < -1)
        return -1;
    if (p->window_left < -1 || (p->window_left >= 0 && p->mask == ORC_MASK_NONE))
        return -1;
    for (int b = 0; b < p->B; ++b)
        if (p->cu_q[b + 1] < p->cu_q[b] || p->cu_k[b + 1] < p->cu_k[b])
            return -1;
    return 0;
}

static int seq_len_q(const orc_problem *p, int b) { return p->cu_q[b + 1] - p->cu_q[b]; }
/* Keys of sequence b: its cu_seqlens slot, shortened to seqused_k[b] when the slot is
 * padded ([P2] Technical details: padded cu_seqlens). */
static int seq_len_k(const orc_problem *p, int b)
{
    int n = p->cu_k[b + 1] - p->cu_k[b];
    if (p->seqused_k && p->seqused_k[b] < n)
        n = p->seqused_k[b] < 0 ? 0 : p->seqused_k[b];
    return n;
}

/* Query position offset added before the causal comparison: 0 for plain causal. */
static int offset_of(const orc_problem *p)
{
    return p->mask == ORC_MASK_PREFIX_CAUSAL ? p->prefix_offset : 0;
}

/* [P1] Technical details: lastValid is last_valid_kv_index, default seq_len_k - 1.
 * For packed sequences it is also capped at the sequence's own last key. */
int orc_last_valid(const orc_problem *p, int b)
{
    int last = seq_len_k(p, b) - 1;
    if (p->last_valid_kv_index >= 0 && p->last_valid_kv_index < last)
        last = p->last_valid_kv_index;
    return last;
}

/* Key j is visible to query q when it is a valid key and, under a causal mask, not
 * after q + prefix_offset; with a sliding window ([P2] Technical details: the forced
 * split honours the caller's window) also not before q + prefix_offset - window_left. */
int orc_visible(const orc_problem *p, int b, int q, int j)
{
    if (j < 0 || j > orc_last_valid(p, b))
        return 0;
    if (p->mask != ORC_MASK_NONE) {
        long long diag = (long long)q + offset_of(p);
        if ((long long)j > diag)
            return 0;
        if (p->window_left >= 0 && (long long)j < diag - p->window_left)
            return 0;
    }
    return 1;
}

static long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

/* clamp(x, lo, hi) read as min(max(x, lo), hi), so that hi = -1 (no key) wins. */
static long long clamp_ll(long long x, long long lo, long long hi)
{
    if (x < lo) x = lo;
    if (x > hi) x = hi;
    return x;
}

/* The last key index that a split partition must cover for "row" (a row, or the
 * last row of an M block): [P1] rowLast = clamp(q + prefix_offset, 0, lastValid)
 * under causal / prefix-causal masks; lastValid without a mask (one count per
 * batch-head). Returns -1 when the sequence has no key. */
static long long covered_last(const orc_problem *p, int b, long long row)
{
    long long last_valid = orc_last_valid(p, b);
    if (last_valid < 0)
        return -1;
    if (p->mask == ORC_MASK_NONE)
        return last_valid;
    return clamp_ll(row + offset_of(p), 0, last_valid);
}

/* [P1] Per-row valid-split counts:
 *   keysPerSplit = nPerBlock * ceil(ceil((rowLast + 1) / nPerBlock) / split_kv)
 *   count        = ceil((rowLast + 1) / keysPerSplit)
 * A sequence with no key has nothing to divide; its rows get count 1 ([P1]
 * review notes: the count is always >= 1). */
int orc_split_counts(const orc_problem *p, int32_t *counts)
{
    if (orc_check_problem(p) || !counts)
        return -1;
    for (int b = 0; b < p->B; ++b) {
        for (int q = 0; q < seq_len_q(p, b); ++q) {
            long long row_last = covered_last(p, b, q);
            long long c = 1;
            if (row_last >= 0) {
                long long n = row_last + 1;
                long long keys_per_split =
                    (long long)p->n_per_block * ceil_div(ceil_div(n, p->n_per_block), p->split_kv);
                c = ceil_div(n, keys_per_split);
            }
            counts[p->cu_q[b] + q] = (int32_t)c;
        }
    }
    return 0;
}

/* [P1] Technical details, kernel partition: an M block's keys are split by the
 * block's last row: the block's key tiles 0 .. nT-1 (nT = ceil((blockLast + 1) / nPerBlock)) are
 * dealt out in runs of itersPerBlock = ceil(nT / split_kv) tiles, split s taking
 * tiles [s * itersPerBlock, (s + 1) * itersPerBlock). Keys after blockLast are
 * masked for every row of the block, so the range stops at blockLast + 1. */
int orc_split_range(const orc_problem *p, int b, int q, int s, int *k_begin, int *k_end)
{
    if (orc_check_problem(p) || b < 0 || b >= p->B || q < 0 || q >= seq_len_q(p, b) ||
        s < 0 || s >= p->split_kv || !k_begin || !k_end)
        return -1;
    long long sq = seq_len_q(p, b);
    long long first_row = (q / p->block_m) * (long long)p->block_m;
    long long last_row = first_row + p->block_m - 1;
    if (last_row > sq - 1)
        last_row = sq - 1;
    long long block_last = covered_last(p, b, last_row);
    *k_begin = *k_end = 0;
    if (block_last < 0)
        return 0;
    long long n_tiles = ceil_div(block_last + 1, p->n_per_block);
    long long iters = ceil_div(n_tiles, p->split_kv);
    long long t0 = (long long)s * iters, t1 = t0 + iters;
    if (t1 > n_tiles) t1 = n_tiles;
    if (t0 >= t1)
        return 0;
    long long kb = t0 * p->n_per_block, ke = t1 * p->n_per_block;
    if (ke > block_last + 1) ke = block_last + 1;
    *k_begin = (int)kb;
    *k_end = (int)ke;
    return 0;
}

int orc_split_ranges(const orc_problem *p, int32_t *k_begin, int32_t *k_end)
{
    if (orc_check_problem(p) || !k_begin || !k_end)
        return -1;
    for (int b = 0; b < p->B; ++b)
        for (int q = 0; q < seq_len_q(p, b); ++q)
            for (int s = 0; s < p->split_kv; ++s) {
                int kb, ke;
                orc_split_range(p, b, q, s, &kb, &ke);
                int64_t slot = ((int64_t)p->cu_q[b] + q) * p->split_kv + s;
                k_begin[slot] = kb;
                k_end[slot] = ke;
            }
    return 0;
}

/* ------------------------------------------------------- attention, direct */

/* Softmax attention of query row (b, q, h) over the visible keys with index in
 * [kb, ke):  s_j = scale * q.k_j,  O = sum_j softmax(s)_j v_j,
 * LSE = log sum_j exp(s_j) (natural log of the scaled scores). No visible key:
 * O = 0 and LSE = -inf. "scores" has room for ke - kb doubles. */
static void attend(const orc_problem *p, orc_array Q, orc_array K, orc_array V, int b, int q,
                   int h, int kb, int ke, double *scores, double *o, double *lse)
{
    const int H = p->H, dqk = p->d_qk, dv = p->d_v;
    const int64_t qrow = (int64_t)p->cu_q[b] + q;
    double m = -INFINITY;
    int any = 0;
    for (int j = kb; j < ke; ++j) {
        if (!orc_visible(p, b, q, j)) {
            scores[j - kb] = -INFINITY;
            continue;
        }
        const int64_t krow = (int64_t)p->cu_k[b] + j;
        double dot = 0.0;
        for (int d = 0; d < dqk; ++d)
            dot += orc_load(Q, (qrow * H + h) * dqk + d) * orc_load(K, (krow * H + h) * dqk + d);
        double sc = p->scale * dot;
        scores[j - kb] = sc;
        if (sc > m) m = sc;
        any = 1;
    }
    for (int d = 0; d < dv; ++d)
        o[d] = 0.0;
    if (!any) {
        *lse = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int j = kb; j < ke; ++j) {
        if (scores[j - kb] == -INFINITY)
            continue;
        double w = exp(scores[j - kb] - m);
        const int64_t krow = (int64_t)p->cu_k[b] + j;
        z += w;
        for (int d = 0; d < dv; ++d)
            o[d] += w * orc_load(V, (krow * H + h) * dv + d);
    }
    for (int d = 0; d < dv; ++d)
        o[d] /= z;
    *lse = m + log(z);
}

/* sequence holding packed row r */
static int seq_of_row(const orc_problem *p, int r)
{
    int lo = 0, hi = p->B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (p->cu_q[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

typedef struct {
    const orc_problem *p;
    orc_array q, k, v;
    const int32_t *rows;
    int n_rows, split, tid, nthreads, max_sk;
    double *out, *lse;      /* split == 0 */
    double *o_part, *l_part;/* split == 1 */
} orc_job;

static void *orc_worker(void *arg)
{
    orc_job *J = (orc_job *)arg;
    const orc_problem *p = J->p;
    const int H = p->H, dv = p->d_v, S = p->split_kv;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(J->max_sk > 0 ? J->max_sk : 1));
    if (!scores)
        return (void *)1;
    for (int i = J->tid; i < J->n_rows; i += J->nthreads) {
        int r = J->rows[i];
        int b = seq_of_row(p, r);
        int qpos = r - p->cu_q[b];
        for (int h = 0; h < H; ++h) {
            if (!J->split) {
                attend(p, J->q, J->k, J->v, b, qpos, h, 0, seq_len_k(p, b), scores,
                       J->out + ((int64_t)i * H + h) * dv, J->lse + (int64_t)i * H + h);
            } else {
                for (int s = 0; s < S; ++s) {
                    int kb, ke;
                    orc_split_range(p, b, qpos, s, &kb, &ke);
                    int64_t slot = ((int64_t)i * H + h) * S + s;
                    attend(p, J->q, J->k, J->v, b, qpos, h, kb, ke, scores,
                           J->o_part + slot * dv, J->l_part + slot);
                }
            }
        }
    }
    free(scores);
    return NULL;
}

static int run_rows(const orc_problem *p, orc_array q, orc_array k, orc_array v,
                    const int32_t *rows, int n_rows, int split, double *a, double *c, int nthreads)
{
    if (orc_check_problem(p) || n_rows < 0 || (n_rows > 0 && (!rows || !a || !c)))
        return -1;
    int total_q = p->cu_q[p->B];
    int max_sk = 0;
    for (int i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_q)
            return -1;
    for (int b = 0; b < p->B; ++b)
        if (seq_len_k(p, b) > max_sk) max_sk = seq_len_k(p, b);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_rows) nthreads = n_rows > 0 ? n_rows : 1;
    orc_job *jobs = (orc_job *)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        orc_job J = {p, q, k, v, rows, n_rows, split, t, nthreads, max_sk,
                     split ? NULL : a, split ? NULL : c, split ? a : NULL, split ? c : NULL};
        jobs[t] = J;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, orc_worker, &jobs[t]) != 0) { rc = -2; break; }
        started = t;
    }
    if (rc == 0 && orc_worker(&jobs[0]) != NULL) rc = -2;
    for (int t = 1; t <= started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = -2;
    }
    free(jobs);
    free(th);
    return rc;
}

int orc_attention(const orc_problem *p, orc_array q, orc_array k, orc_array v,
                  const int32_t *rows, int n_rows, double *out, double *lse, int nthreads)
{
    return run_rows(p, q, k, v, rows, n_rows, 0, out, lse, nthreads);
}

int orc_partials(const orc_problem *p, orc_array q, orc_array k, orc_array v,
                 const int32_t *rows, int n_rows, double *o_part, double *l_part, int nthreads)
{
    return run_rows(p, q, k, v, rows, n_rows, 1, o_part, l_part, nthreads);
}

/* ------------------------------------------------------------------ merge */

/* [P1] NaN-safe merge, per row and head, over the splits s < count (split s is
 * valid for a row when s < count; the others never enter the sums):
 *   m   = max(max_s L_s, lowest finite)
 *   w_s = exp(L_s - m)
 *   O   = sum_s(w_s * O_s) / max(sum_s w_s, 1)
 * The final log-sum-exp is m + log(sum_s w_s), or -inf when every valid split is
 * empty (the sum is then 0). */
int orc_merge(int n_rows, int H, int S, int d_v, const double *o_part, const double *l_part,
              const int32_t *counts, double *out, double *lse)
{
    if (n_rows < 0 || H <= 0 || S <= 0 || d_v <= 0)
        return -1;
    if (n_rows > 0 && (!o_part || !l_part || !counts || !out || !lse))
        return -1;
    for (int i = 0; i < n_rows; ++i) {
        int count = counts[i];
        if (count < 1 || count > S)
            return -1;
        for (int h = 0; h < H; ++h) {
            const int64_t slot0 = ((int64_t)i * H + h) * S;
            double m = -DBL_MAX;                     /* lowest finite double */
            for (int s = 0; s < count; ++s)
                if (l_part[slot0 + s] > m) m = l_part[slot0 + s];
            double wsum = 0.0;
            double *o = out + ((int64_t)i * H + h) * d_v;
            for (int d = 0; d < d_v; ++d)
                o[d] = 0.0;
            for (int s = 0; s < count; ++s) {
                double w = exp(l_part[slot0 + s] - m);
                wsum += w;
                for (int d = 0; d < d_v; ++d)
                    o[d] += w * o_part[(slot0 + s) * d_v + d];
            }
            double denom = wsum > 1.0 ? wsum : 1.0;
            for (int d = 0; d < d_v; ++d)
                o[d] /= denom;
            lse[(int64_t)i * H + h] = wsum > 0.0 ? m + log(wsum) : -INFINITY;
        }
    }
    return 0;
}
