/*
 * vsd_oracle.c -- plain, slow, fp64 CPU oracle for verification-guided sparse
 * self-speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library; the only things the two sides have in common are the data layouts,
 * which are the public definition of the inputs.
 *
 * Sources (page titles and sections):
 *   [Vegas]  "Vegas - verification-guided sparse attention for self-speculative
 *            decoding" (technical summary), sec. 2 "Methodology" (verification
 *            phase, KV selection, drafting phase), sec. 2.A "Aggregated attention
 *            logit selection" (the selection equation), sec. 2.B "Collect-2-Query",
 *            sec. 3 "Implementation" (pre-softmax logits written to HBM; draft
 *            attention is paged attention with page size 1 over the selected
 *            token indices).
 *   [Dustin] "Dustin" (technical summary), "Methodology" sec. 1 "Hybrid attention
 *            aggregation" (a few attention-sink prefix tokens and a local window of
 *            recent tokens are always protected; the rest of the budget is filled
 *            by score).
 *
 * Every floating-point step is done in double precision.  bf16 inputs are widened
 * exactly (a bf16 value is the top half of an IEEE binary32).
 *
 * Data layouts (element offsets; all arrays dense, row-major):
 *   q verify     [B][R][Hq][d]            bf16 bits
 *   q decode     [B][Hq][d]               bf16 bits
 *   k/v cache    [num_blocks][Hkv][page][d] bf16 bits
 *   block_table  [B][max_blocks]          logical page p of sequence b lives in
 *                                         physical block block_table[b][p]
 *   logits       [B][2][Hq][P_max]        pre-softmax (scaled) logits, j < P_b
 *                [B][R][Hq][P_max]        (every verify row: oracle_verify_all_rows)
 *   partial      [B][Hkv][P_max]          sum over the two collected rows and the
 *                                         query heads of one KV group
 *   score        [n_rows][P_max]          sum over rows and all query heads
 *   idx          [n_rows][k]              selected prefix positions, ascending
 *
 * Readings of the pages taken here (where they are silent):
 *   - logits are scaled by `scale` (the value softmax consumes);
 *   - query head h reads KV head h / (Hq / Hkv) (contiguous groups);
 *   - verify row t of sequence b sees keys 0 .. P_b + t (causal inside the block);
 *   - the score sums the two collected rows only and all query heads;
 *   - only prefix positions j < P_b are scored and selected;
 *   - the budget k counts the protected tokens; overlapping sink and recent ranges
 *     count once; ties in the score go to the lower position.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_BAD_INDEX -2
#define ORACLE_NO_MEMORY -3

static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Address of the d-vector of logical token j, KV head g, of sequence b in a paged
 * cache, or NULL if the block table points outside the cache.  [Vegas] sec. 3:
 * the cache is paged; a page holds `page` consecutive tokens. */
static const uint16_t *kv_row(const uint16_t *cache, const int32_t *block_table, int b,
                              int max_blocks, int num_blocks, int Hkv, int page, int d,
                              int j, int g) {
    int logical_page = j / page;
    if (logical_page >= max_blocks) return NULL;
    int32_t blk = block_table[(size_t)b * max_blocks + logical_page];
    if (blk < 0 || blk >= num_blocks) return NULL;
    size_t off = (((size_t)blk * Hkv + g) * page + (size_t)(j % page)) * d;
    return cache + off;
}

/* Softmax attention of one query vector over a list of key positions, in the order
 * given (a position listed twice is attended twice).  Writes the attention output
 * (d values) and, if z_out is not NULL, the scaled logits z_n = scale * q . K_{pos[n]}.
 * [Vegas] sec. 2, verification phase: full attention computes the logit of every
 * KV entry; drafting phase: the same attention restricted to selected entries. */
static int attend(const double *qv, int d, const int *pos, int n_pos, const uint16_t *k_cache,
                  const uint16_t *v_cache, const int32_t *block_table, int b, int max_blocks,
                  int num_blocks, int Hkv, int page, int g, double scale, double *o,
                  double *z_out) {
    double *z = (double *)malloc(sizeof(double) * (size_t)(n_pos > 0 ? n_pos : 1));
    if (!z) return ORACLE_NO_MEMORY;
    double zmax = -INFINITY;
    for (int n = 0; n < n_pos; ++n) {
        const uint16_t *kr = kv_row(k_cache, block_table, b, max_blocks, num_blocks, Hkv,
                                    page, d, pos[n], g);
        if (!kr) { free(z); return ORACLE_BAD_INDEX; }
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qv[c] * bf16_to_double(kr[c]);
        z[n] = scale * dot;
        if (z[n] > zmax) zmax = z[n];
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    double denom = 0.0;
    for (int n = 0; n < n_pos; ++n) {
        double p = exp(z[n] - zmax);
        denom += p;
        const uint16_t *vr = kv_row(v_cache, block_table, b, max_blocks, num_blocks, Hkv,
                                    page, d, pos[n], g);
        if (!vr) { free(z); return ORACLE_BAD_INDEX; }
        for (int c = 0; c < d; ++c) o[c] += p * bf16_to_double(vr[c]);
    }
    if (n_pos > 0)
        for (int c = 0; c < d; ++c) o[c] /= denom;
    if (z_out)
        for (int n = 0; n < n_pos; ++n) z_out[n] = z[n];
    free(z);
    return ORACLE_OK;
}

/*
 * Verification pass with Collect-2-Query.
 *   [Vegas] sec. 2, verification phase: the gamma+1 verify rows attend the whole
 *   cache with full attention.  sec. 2.B: only the logits of the first draft token
 *   and of the bonus token are collected (rows row0 and row1 of the block, which
 *   are 0 and gamma for the plain reading).  sec. 3: the collected values are the
 *   pre-softmax logits, written to memory.
 * Outputs: out[b][t][h][:] (attention output), logits[b][c][h][j] for j < P_b,
 * partial[b][g][j] = sum over c in {0,1} and h in group g of logits[b][c][h][j].
 * logits / partial may be NULL.
 */
int oracle_verify(int B, int Hq, int Hkv, int d, int page, int max_blocks, int num_blocks,
                  int R, const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                  const int32_t *block_table, const int32_t *prefix_len, int row0, int row1,
                  int P_max, double scale, double *logits, double *partial, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page <= 0 || R <= 0)
        return ORACLE_BAD_ARG;
    if ((logits || partial) && (row0 < 0 || row0 >= R || row1 < 0 || row1 >= R))
        return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    const int n_items = B * R * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int item = 0; item < n_items; ++item) {
        int b = item / (R * Hq);
        int t = (item / Hq) % R;
        int h = item % Hq;
        int g = h / G;
        int P = prefix_len[b];
        if (P < 0 || P > P_max) { status = ORACLE_BAD_ARG; continue; }
        int n_keys = P + t + 1; /* causal inside the verify block */
        int *pos = (int *)malloc(sizeof(int) * (size_t)n_keys);
        double *z = (double *)malloc(sizeof(double) * (size_t)n_keys);
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!pos || !z || !qv || !o) {
            status = ORACLE_NO_MEMORY;
        } else {
            for (int j = 0; j < n_keys; ++j) pos[j] = j;
            const uint16_t *qr = q + (((size_t)b * R + t) * Hq + h) * d;
            for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(qr[c]);
            int rc = attend(qv, d, pos, n_keys, k_cache, v_cache, block_table, b, max_blocks,
                            num_blocks, Hkv, page, g, scale, o, z);
            if (rc != ORACLE_OK) {
                status = rc;
            } else {
                double *dst = out + (((size_t)b * R + t) * Hq + h) * d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
                if (logits) {
                    for (int which = 0; which < 2; ++which) {
                        int row = which == 0 ? row0 : row1;
                        if (row != t) continue;
                        double *lrow = logits + (((size_t)b * 2 + which) * Hq + h) * P_max;
                        for (int j = 0; j < P; ++j) lrow[j] = z[j];
                    }
                }
            }
        }
        free(pos); free(z); free(qv); free(o);
    }
    if (status != ORACLE_OK || !partial) return status;
    if (!logits) return ORACLE_BAD_ARG; /* the partial sums are defined from the logits */
    /* [Vegas] sec. 2.A: the selection objective sums logits over draft rows and
     * query heads; the per-KV-group partial sum is that sum restricted to the
     * query heads of one group. */
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b];
        for (int g = 0; g < Hkv; ++g) {
            double *prow = partial + ((size_t)b * Hkv + g) * P_max;
            for (int j = 0; j < P; ++j) {
                double s = 0.0;
                for (int which = 0; which < 2; ++which)
                    for (int h = g * G; h < (g + 1) * G; ++h)
                        s += logits[(((size_t)b * 2 + which) * Hq + h) * P_max + j];
                prow[j] = s;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Verification with every verify row collected (the selection equation as printed).
 *   [Vegas] sec. 2.A: the objective sums the logits over the draft rows t = 1..gamma+1
 *   of the verification block and over the query heads; sec. 2.B (Collect-2-Query)
 *   keeps two of those rows, which is what oracle_verify collects.  This variant keeps
 *   all R of them, the reference Collect-2-Query is measured against.
 * Outputs: out[b][t][h][:] as oracle_verify; logits[b][t][h][j] for every row t and
 * j < P_b; partial[b][g][j] = sum over t < R and h in group g of logits[b][t][h][j].
 * logits / partial may be NULL (partial needs logits).
 */
int oracle_verify_all_rows(int B, int Hq, int Hkv, int d, int page, int max_blocks,
                           int num_blocks, int R, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_table,
                           const int32_t *prefix_len, int P_max, double scale, double *logits,
                           double *partial, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page <= 0 || R <= 0)
        return ORACLE_BAD_ARG;
    if (partial && !logits) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    const int n_items = B * R * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int item = 0; item < n_items; ++item) {
        int b = item / (R * Hq);
        int t = (item / Hq) % R;
        int h = item % Hq;
        int g = h / G;
        int P = prefix_len[b];
        if (P < 0 || P > P_max) { status = ORACLE_BAD_ARG; continue; }
        int n_keys = P + t + 1;
        int *pos = (int *)malloc(sizeof(int) * (size_t)n_keys);
        double *z = (double *)malloc(sizeof(double) * (size_t)n_keys);
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!pos || !z || !qv || !o) {
            status = ORACLE_NO_MEMORY;
        } else {
            for (int j = 0; j < n_keys; ++j) pos[j] = j;
            const uint16_t *qr = q + (((size_t)b * R + t) * Hq + h) * d;
            for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(qr[c]);
            int rc = attend(qv, d, pos, n_keys, k_cache, v_cache, block_table, b, max_blocks,
                            num_blocks, Hkv, page, g, scale, o, z);
            if (rc != ORACLE_OK) {
                status = rc;
            } else {
                double *dst = out + (((size_t)b * R + t) * Hq + h) * d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
                if (logits) {
                    double *lrow = logits + (((size_t)b * R + t) * Hq + h) * P_max;
                    for (int j = 0; j < P; ++j) lrow[j] = z[j];
                }
            }
        }
        free(pos); free(z); free(qv); free(o);
    }
    if (status != ORACLE_OK || !partial) return status;
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b];
        for (int g = 0; g < Hkv; ++g) {
            double *prow = partial + ((size_t)b * Hkv + g) * P_max;
            for (int j = 0; j < P; ++j) {
                double s = 0.0;
                for (int t = 0; t < R; ++t)
                    for (int h = g * G; h < (g + 1) * G; ++h)
                        s += logits[(((size_t)b * R + t) * Hq + h) * P_max + j];
                prow[j] = s;
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Aggregated score of every prefix position from the collected logits.
 *   [Vegas] sec. 2.A: the selected set maximises the logits summed over draft rows
 *   t and query heads h; with Collect-2-Query (sec. 2.B) the rows are the two
 *   collected ones.  score[b][j] = sum_c sum_h logits[b][c][h][j], j < P_b.
 */
int oracle_score_from_logits(int B, int Hq, int P_max, const double *logits,
                             const int32_t *prefix_len, double *score) {
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b];
        if (P < 0 || P > P_max) return ORACLE_BAD_ARG;
        for (int j = 0; j < P; ++j) {
            double s = 0.0;
            for (int which = 0; which < 2; ++which)
                for (int h = 0; h < Hq; ++h)
                    s += logits[(((size_t)b * 2 + which) * Hq + h) * P_max + j];
            score[(size_t)b * P_max + j] = s;
        }
    }
    return ORACLE_OK;
}

/* Score of every prefix position from per-KV-group partial sums: the same total
 * as oracle_score_from_logits, grouped by KV head. */
int oracle_score_from_partials(int n_rows, int Hkv, int P_max, const double *partial,
                               const int32_t *prefix_len, double *score) {
    for (int r = 0; r < n_rows; ++r) {
        int P = prefix_len[r];
        if (P < 0 || P > P_max) return ORACLE_BAD_ARG;
        for (int j = 0; j < P; ++j) {
            double s = 0.0;
            for (int g = 0; g < Hkv; ++g) s += partial[((size_t)r * Hkv + g) * P_max + j];
            score[(size_t)r * P_max + j] = s;
        }
    }
    return ORACLE_OK;
}

typedef struct {
    double s;
    int j;
} scored_pos;

/* Order for the budget fill: higher score first, lower position first on ties. */
static int by_score_then_position(const void *a, const void *b) {
    const scored_pos *x = (const scored_pos *)a;
    const scored_pos *y = (const scored_pos *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

static int by_int(const void *a, const void *b) {
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

/*
 * Budgeted top-k with protected sink and recent tokens.
 *   [Vegas] sec. 2.A: T = argmax over subsets T of the prefix with |T| = k of the
 *   summed logits; the objective is a sum of per-position scores, so the maximiser
 *   is the k highest-scoring positions.
 *   [Dustin] Methodology sec. 1: a few attention-sink prefix tokens and a local
 *   window of recent tokens are protected first; the rest of the budget is filled
 *   by score.
 * For each row r with prefix length P:
 *   S  = [0, min(n_sink, P))  U  [max(0, P - n_recent), P)
 *   n  = min(k, P);  fill n - |S| positions from the rest by (score desc, j asc)
 *   idx[r][0 .. n) = S U fill, ascending;  n_sel[r] = n.
 * Requires n_sink + n_recent <= k.
 */
int oracle_select(int n_rows, int P_max, const double *score, const int32_t *prefix_len,
                  int k, int n_sink, int n_recent, int32_t *idx, int32_t *n_sel) {
    if (k < 0 || n_sink < 0 || n_recent < 0 || n_sink + n_recent > k) return ORACLE_BAD_ARG;
    for (int r = 0; r < n_rows; ++r) {
        int P = prefix_len[r];
        if (P < 0 || P > P_max) return ORACLE_BAD_ARG;
        int n = k < P ? k : P;
        int sink_end = n_sink < P ? n_sink : P;
        int recent_begin = P - n_recent > 0 ? P - n_recent : 0;
        int *chosen = (int *)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
        scored_pos *rest = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(P > 0 ? P : 1));
        if (!chosen || !rest) { free(chosen); free(rest); return ORACLE_NO_MEMORY; }
        int n_chosen = 0, n_rest = 0;
        for (int j = 0; j < P; ++j) {
            int protected_pos = (j < sink_end) || (j >= recent_begin);
            if (protected_pos) {
                chosen[n_chosen++] = j;
            } else {
                rest[n_rest].s = score[(size_t)r * P_max + j];
                rest[n_rest].j = j;
                ++n_rest;
            }
        }
        if (n_chosen > n) { free(chosen); free(rest); return ORACLE_BAD_ARG; }
        qsort(rest, (size_t)n_rest, sizeof(scored_pos), by_score_then_position);
        for (int m = 0; n_chosen < n; ++m) chosen[n_chosen++] = rest[m].j;
        qsort(chosen, (size_t)n_chosen, sizeof(int), by_int);
        for (int m = 0; m < n_chosen; ++m) idx[(size_t)r * k + m] = chosen[m];
        n_sel[r] = n_chosen;
        free(chosen);
        free(rest);
    }
    return ORACLE_OK;
}

/*
 * Hybrid budget with two signals.
 *   [Dustin] Methodology sec. 1 (hybrid attention aggregation): after the
 *   attention-sink prefix and the local window of recent tokens are protected, the
 *   rest of the budget is allocated hierarchically: first the top-m tokens by the
 *   draft-lookahead signal, then the most relevant remaining tokens by the
 *   target-historical signal.
 * For each row r with prefix length P (n = min(k, P), S as in oracle_select):
 *   D  = the min(m, n - |S|) positions outside S with the highest draft score
 *        (ties: lower position first)
 *   T' = the n - |S| - |D| positions outside S and D with the highest target score
 *        (ties: lower position first)
 *   idx[r][0 .. n) = S U D U T', ascending;  n_sel[r] = n.
 * Requires n_sink + n_recent <= k and m >= 0.
 */
int oracle_select_hybrid(int n_rows, int P_max, const double *score_target,
                         const double *score_draft, const int32_t *prefix_len, int k, int m,
                         int n_sink, int n_recent, int32_t *idx, int32_t *n_sel) {
    if (k < 0 || m < 0 || n_sink < 0 || n_recent < 0 || n_sink + n_recent > k)
        return ORACLE_BAD_ARG;
    for (int r = 0; r < n_rows; ++r) {
        int P = prefix_len[r];
        if (P < 0 || P > P_max) return ORACLE_BAD_ARG;
        int n = k < P ? k : P;
        int sink_end = n_sink < P ? n_sink : P;
        int recent_begin = P - n_recent > 0 ? P - n_recent : 0;
        int *chosen = (int *)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
        char *taken = (char *)calloc((size_t)(P > 0 ? P : 1), 1);
        scored_pos *rest = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(P > 0 ? P : 1));
        if (!chosen || !taken || !rest) {
            free(chosen); free(taken); free(rest);
            return ORACLE_NO_MEMORY;
        }
        int n_chosen = 0;
        for (int j = 0; j < P; ++j)
            if (j < sink_end || j >= recent_begin) { chosen[n_chosen++] = j; taken[j] = 1; }
        if (n_chosen > n) { free(chosen); free(taken); free(rest); return ORACLE_BAD_ARG; }
        /* draft signal first, at most m of them */
        int n_rest = 0;
        for (int j = 0; j < P; ++j)
            if (!taken[j]) { rest[n_rest].s = score_draft[(size_t)r * P_max + j]; rest[n_rest].j = j; ++n_rest; }
        qsort(rest, (size_t)n_rest, sizeof(scored_pos), by_score_then_position);
        int n_draft = n - n_chosen < m ? n - n_chosen : m;
        for (int q = 0; q < n_draft; ++q) { chosen[n_chosen++] = rest[q].j; taken[rest[q].j] = 1; }
        /* then the target signal over what is left */
        n_rest = 0;
        for (int j = 0; j < P; ++j)
            if (!taken[j]) { rest[n_rest].s = score_target[(size_t)r * P_max + j]; rest[n_rest].j = j; ++n_rest; }
        qsort(rest, (size_t)n_rest, sizeof(scored_pos), by_score_then_position);
        for (int q = 0; n_chosen < n; ++q) chosen[n_chosen++] = rest[q].j;
        qsort(chosen, (size_t)n_chosen, sizeof(int), by_int);
        for (int q = 0; q < n_chosen; ++q) idx[(size_t)r * k + q] = chosen[q];
        n_sel[r] = n_chosen;
        free(chosen); free(taken); free(rest);
    }
    return ORACLE_OK;
}

/*
 * Per-KV-group partial scores restricted to a subset of query heads.
 *   [Dustin] Methodology sec. 2 (semantic retrieval heads): online, the importance
 *   computation is restricted to the few heads identified offline.
 * partial[b][g][j] = sum over the collected rows c and the heads h of group g with
 * head_mask[h] != 0 of logits[b][c][h][j], j < P_b (logits [B][C][Hq][P_max]).
 */
int oracle_partial_masked(int B, int C, int Hq, int Hkv, int P_max, const double *logits,
                          const int32_t *prefix_len, const uint8_t *head_mask,
                          double *partial) {
    if (B < 0 || C <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b];
        if (P < 0 || P > P_max) return ORACLE_BAD_ARG;
        for (int g = 0; g < Hkv; ++g)
            for (int j = 0; j < P; ++j) {
                double s = 0.0;
                for (int c = 0; c < C; ++c)
                    for (int h = g * G; h < (g + 1) * G; ++h)
                        if (head_mask[h]) s += logits[(((size_t)b * C + c) * Hq + h) * P_max + j];
                partial[((size_t)b * Hkv + g) * P_max + j] = s;
            }
    }
    return ORACLE_OK;
}

/*
 * Per-query block top-k (the sparse-verification summary, "Sparse Verification
 * Engine", attention sparsity: each query keeps only its top-k keys/values in
 * structured blocks, chosen by a cheap relevance score).  Reading taken here: the
 * blocks are the 16-token pages of the prefix, the cheap score of block beta for a
 * query is the scaled dot product with the block's mean key
 *   kbar[b][beta][g][:] = mean over j in block beta, j < P_b, of K[b][j][g][:]
 *   r[b][t][h][beta]    = scale * <q[b][t][h][:], kbar[b][beta][h/G][:]>
 * and each (b, t, h) keeps the kb blocks with the highest r (ties: lower block
 * first), listed in ascending block order: blocks[b][t][h][0 .. min(kb, nblk_b)),
 * nblk_b = ceil(P_b / page); unused entries -1.
 */
int oracle_block_topk(int B, int Hq, int Hkv, int d, int page, int max_blocks, int num_blocks,
                      int R, const uint16_t *q, const uint16_t *k_cache,
                      const int32_t *block_table, const int32_t *prefix_len, int kb,
                      double scale, double *scores_out, int P_blk_max, int32_t *blocks) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page <= 0 || R <= 0 ||
        kb <= 0)
        return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    const int n_items = B * R * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int item = 0; item < n_items; ++item) {
        int b = item / (R * Hq);
        int t = (item / Hq) % R;
        int h = item % Hq;
        int g = h / G;
        int P = prefix_len[b];
        int nblk = (P + page - 1) / page;
        if (P < 0 || nblk > P_blk_max) { status = ORACLE_BAD_ARG; continue; }
        scored_pos *sc = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(nblk > 0 ? nblk : 1));
        double *kbar = (double *)malloc(sizeof(double) * (size_t)d);
        int *chosen = (int *)malloc(sizeof(int) * (size_t)kb);
        if (!sc || !kbar || !chosen) {
            status = ORACLE_NO_MEMORY;
        } else {
            const uint16_t *qr = q + (((size_t)b * R + t) * Hq + h) * d;
            for (int beta = 0; beta < nblk; ++beta) {
                int j0 = beta * page, j1 = j0 + page < P ? j0 + page : P;
                for (int c = 0; c < d; ++c) kbar[c] = 0.0;
                int bad = 0;
                for (int j = j0; j < j1; ++j) {
                    const uint16_t *kr = kv_row(k_cache, block_table, b, max_blocks, num_blocks,
                                                Hkv, page, d, j, g);
                    if (!kr) { bad = 1; break; }
                    for (int c = 0; c < d; ++c) kbar[c] += bf16_to_double(kr[c]);
                }
                if (bad) { status = ORACLE_BAD_INDEX; nblk = 0; break; }
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += bf16_to_double(qr[c]) * (kbar[c] / (j1 - j0));
                sc[beta].s = scale * dot;
                sc[beta].j = beta;
                if (scores_out)
                    scores_out[(((size_t)b * R + t) * Hq + h) * P_blk_max + beta] = sc[beta].s;
            }
            qsort(sc, (size_t)nblk, sizeof(scored_pos), by_score_then_position);
            int n = kb < nblk ? kb : nblk;
            for (int m = 0; m < n; ++m) chosen[m] = sc[m].j;
            qsort(chosen, (size_t)n, sizeof(int), by_int);
            int32_t *dst = blocks + (((size_t)b * R + t) * Hq + h) * kb;
            for (int m = 0; m < kb; ++m) dst[m] = m < n ? chosen[m] : -1;
        }
        free(sc); free(kbar); free(chosen);
    }
    return status;
}

/*
 * Sparse draft-step attention.
 *   [Vegas] sec. 2, drafting phase: the draft step uses attention restricted to the
 *   selected KV entries.  sec. 3: this is paged attention with page size 1 whose
 *   page indices are the selected token indices.  Tokens written after the
 *   selection (positions tail_start .. seq_len-1) are attended densely.
 * For every b, h: attended positions = idx[b][0 .. n_sel[b]) followed by
 * tail_start[b] .. seq_len[b]-1; out[b][h][:] = softmax attention over them.
 */
int oracle_sparse_decode(int B, int Hq, int Hkv, int d, int page, int max_blocks,
                         int num_blocks, const uint16_t *q, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table,
                         const int32_t *idx, const int32_t *n_sel, int k_max,
                         const int32_t *tail_start, const int32_t *seq_len, double scale,
                         double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page <= 0 || k_max < 0)
        return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    const int n_items = B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int item = 0; item < n_items; ++item) {
        int b = item / Hq;
        int h = item % Hq;
        int g = h / G;
        int ns = n_sel ? n_sel[b] : 0;
        int t0 = tail_start ? tail_start[b] : 0;
        int t1 = seq_len[b];
        if (ns < 0 || ns > k_max || t0 < 0 || t1 < t0) { status = ORACLE_BAD_ARG; continue; }
        int n_pos = ns + (t1 - t0);
        int *pos = (int *)malloc(sizeof(int) * (size_t)(n_pos > 0 ? n_pos : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!pos || !qv || !o) {
            status = ORACLE_NO_MEMORY;
        } else {
            for (int m = 0; m < ns; ++m) pos[m] = idx[(size_t)b * k_max + m];
            for (int j = t0; j < t1; ++j) pos[ns + (j - t0)] = j;
            const uint16_t *qr = q + ((size_t)b * Hq + h) * d;
            for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(qr[c]);
            int rc = attend(qv, d, pos, n_pos, k_cache, v_cache, block_table, b, max_blocks,
                            num_blocks, Hkv, page, g, scale, o, NULL);
            if (rc != ORACLE_OK) {
                status = rc;
            } else {
                double *dst = out + ((size_t)b * Hq + h) * d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
            }
        }
        free(pos); free(qv); free(o);
    }
    return status;
}

/*
 * Sparse verification.
 *   [Dustin] "Verification workflow", steps 3-4: a compressed target KV cache is
 *   formed from the selected tokens only, and the target model verifies the draft
 *   tokens against that sparse cache.  The draft tokens being verified are the
 *   verify block itself (positions P_b .. P_b + R - 1), causal as in full
 *   verification.
 * For every b, verify row t and head h: attended positions = idx[b][0 .. n_sel[b])
 * followed by P_b .. P_b + t; out[b][t][h][:] = softmax attention over them.
 */
int oracle_sparse_verify(int B, int Hq, int Hkv, int d, int page, int max_blocks,
                         int num_blocks, int R, const uint16_t *q, const uint16_t *k_cache,
                         const uint16_t *v_cache, const int32_t *block_table,
                         const int32_t *prefix_len, const int32_t *idx, const int32_t *n_sel,
                         int k_max, double scale, double *out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page <= 0 || R <= 0 ||
        k_max < 0)
        return ORACLE_BAD_ARG;
    const int G = Hq / Hkv;
    int status = ORACLE_OK;
    const int n_items = B * R * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int item = 0; item < n_items; ++item) {
        int b = item / (R * Hq);
        int t = (item / Hq) % R;
        int h = item % Hq;
        int g = h / G;
        int ns = n_sel ? n_sel[b] : 0;
        int P = prefix_len[b];
        if (ns < 0 || ns > k_max || P < 0) { status = ORACLE_BAD_ARG; continue; }
        int n_pos = ns + t + 1;
        int *pos = (int *)malloc(sizeof(int) * (size_t)n_pos);
        double *qv = (double *)malloc(sizeof(double) * (size_t)d);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!pos || !qv || !o) {
            status = ORACLE_NO_MEMORY;
        } else {
            for (int m = 0; m < ns; ++m) pos[m] = idx[(size_t)b * k_max + m];
            for (int u = 0; u <= t; ++u) pos[ns + u] = P + u;
            const uint16_t *qr = q + (((size_t)b * R + t) * Hq + h) * d;
            for (int c = 0; c < d; ++c) qv[c] = bf16_to_double(qr[c]);
            int rc = attend(qv, d, pos, n_pos, k_cache, v_cache, block_table, b, max_blocks,
                            num_blocks, Hkv, page, g, scale, o, NULL);
            if (rc != ORACLE_OK) {
                status = rc;
            } else {
                double *dst = out + (((size_t)b * R + t) * Hq + h) * d;
                for (int c = 0; c < d; ++c) dst[c] = o[c];
            }
        }
        free(pos); free(qv); free(o);
    }
    return status;
}

/* Number of threads the parallel loops above use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
