/*
 * oracle.h -- plain CPU reference for split-KV attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers. The CUDA library shares no code, header
 * or constant with this file and never loads it.
 *
 * Sources (cited by page title and section):
 *   [P1] "Recombine fully masked split-KV attention partials on the host"
 *        (ROCm/rocmlirTriton pull request 535): Technical details -- per-row
 *        valid-split counts (computeValidSplitKV), per-row mask layout
 *        (createMaskSplitKV), NaN-safe merge (computeFinalAttentionStage), f32
 *        merge for f16/bf16; review notes on the conservativeness argument.
 *   [P2] "[ASM] [HIP] [JIT] [gfx942] Optimize long-context FMHA with split-KV"
 *        (ROCm/aiter pull request 5592): Motivation (packed varlen, D_QK != D_V),
 *        Technical details (num_splits semantics; the forced split honours the
 *        caller's causal mask, window and padded cu_seqlens).
 *
 * All arithmetic is in double precision, starting from the stored (rounded)
 * input values, which are converted to double exactly.
 *
 * Layouts (all contiguous, row-major):
 *   q  [total_q][H][d_qk]    k [total_k][H][d_qk]    v [total_k][H][d_v]
 *   packed row r of sequence b holds query position q = r - cu_q[b].
 *   Results are written for a caller-chosen list of packed rows:
 *   out   [n_rows][H][d_v]      lse    [n_rows][H]
 *   o_part[n_rows][H][S][d_v]   l_part [n_rows][H][S]
 */
#ifndef SPLITKV_ORACLE_H
#define SPLITKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage types of the input arrays */
enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2, ORC_F64 = 3 };
/* mask modes: [P1] Technical details -- plain causal is prefix-causal with offset 0 */
enum { ORC_MASK_NONE = 0, ORC_MASK_CAUSAL = 1, ORC_MASK_PREFIX_CAUSAL = 2 };

typedef struct {
    int B, H, d_qk, d_v;
    const int32_t *cu_q;          /* host int32 [B+1], cu_q[0] = 0 */
    const int32_t *cu_k;          /* host int32 [B+1], cu_k[0] = 0 */
    int mask;                     /* ORC_MASK_* */
    int prefix_offset;            /* used by ORC_MASK_PREFIX_CAUSAL only */
    int last_valid_kv_index;      /* -1: Sk_b - 1; otherwise min(it, Sk_b - 1) */
    int n_per_block;              /* key tile, nPerBlock (> 0) */
    int split_kv;                 /* number of splits S (>= 1) */
    int block_m;                  /* query rows per M block of the kernel partition (> 0) */
    double scale;                 /* softmax scale applied to q.k */
    int window_left;              /* -1: none; else (causal masks only) keys before
                                     q + offset - window_left are not visible */
    const int32_t *seqused_k;     /* NULL, or host int32 [B]: keys of sequence b at or past
                                     seqused_k[b] are padding (not part of the sequence) */
} orc_problem;

typedef struct {
    const void *data;
    int dtype;                    /* ORC_BF16 .. ORC_F64 */
} orc_array;

/* 0 on success, negative on a bad argument. */
int orc_check_problem(const orc_problem *p);

/* Last key a sequence may attend to (lastValid); -1 when the sequence has no key. */
int orc_last_valid(const orc_problem *p, int b);

/* 1 if query position q of sequence b may attend to key j of that sequence. */
int orc_visible(const orc_problem *p, int b, int q, int j);

/* Per packed row valid-split count ([P1] computeValidSplitKV), int32 [total_q]. */
int orc_split_counts(const orc_problem *p, int32_t *counts);

/* Key range [*k_begin, *k_end) of split s for the M block holding query q of
 * sequence b, partitioned by the block's last row ([P1] Technical details and
 * the review notes on itersPerBlock). An empty split gives k_begin == k_end. */
int orc_split_range(const orc_problem *p, int b, int q, int s, int *k_begin, int *k_end);

/* orc_split_range for every packed row and split: k_begin/k_end int32 [total_q][S]. */
int orc_split_ranges(const orc_problem *p, int32_t *k_begin, int32_t *k_end);

/* Unsplit masked softmax attention straight from its definition. */
int orc_attention(const orc_problem *p, orc_array q, orc_array k, orc_array v,
                  const int32_t *rows, int n_rows, double *out, double *lse, int nthreads);

/* Per-split partial outputs O_s and log-sum-exps L_s over the keys of each
 * split's range; a split with no visible key gives O_s = 0, L_s = -inf. */
int orc_partials(const orc_problem *p, orc_array q, orc_array k, orc_array v,
                 const int32_t *rows, int n_rows, double *o_part, double *l_part, int nthreads);

/* NaN-safe merge of S partials with per-row valid-split counts ([P1]
 * computeFinalAttentionStage). Splits s >= counts[r] are never read. */
int orc_merge(int n_rows, int H, int S, int d_v, const double *o_part, const double *l_part,
              const int32_t *counts, double *out, double *lse);

#ifdef __cplusplus
}
#endif
#endif
