/*
 * qsa_oracle.c -- plain, slow CPU oracle for query-sparse-attention block
 * selection.  TEST INFRASTRUCTURE ONLY: the parity tests, the smoke check and
 * the benchmark's CPU-baseline leg call it; the CUDA library never does, and
 * the two share no code.
 *
 * What it computes (written out directly, no blocking, fusion or reordering):
 *
 *   score[q][b] = sum_{h < H} w[q][h] * max(0, sum_{d < D} q[q][h][d] * kblk[b][d])
 *
 * for every block b < n_blocks[q], in IEEE double.  This is the indexer block
 * scorer of "#1091 qsa_select: FP32 tiled block scores below sm_80" (section
 * "What": rows are query x indexer head, the reduction runs over the head
 * dimension K = 128, and the ReLU of each head is weighted and summed per
 * block).  Inputs are read from the same fp32, bf16 or fp8 e4m3 bits the GPU
 * reads and widened exactly (each is a subset of double), so every product is
 * exact in double and the only rounding is in the 128-term and H-term sums.
 *
 * The selection keeps, per query, the k blocks that come first in the order
 * "score descending, then block id ascending", and writes their ids in
 * ascending order, padding with -1 when n < k.  This is the result of the
 * threshold / "above" / tie-budget rule of "#2093 sm_75: the prompt path's
 * top-k with one full read of the scores" (description, step 3) when the
 * tie budget is spent on the lowest block ids, and the ascending-id emit of
 * the same step.  It is done here with a full sort of all n blocks; the sort
 * key (score desc, id asc) is a total order, so the result is the same as a
 * stable sort by score of the blocks listed in id order.
 *
 * The third function, selection attention over the selected blocks, is
 * described above its definition.
 *
 * Parity status: pinned.  The pins (hand-computed fixtures, closed forms,
 * exact-sum cross checks, brute force over all k-subsets) live in the tests.
 *
 * NaN scores are outside the contract (the pages never define their order);
 * -0 and +0 compare equal, so they tie and the lower id wins.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2, ORACLE_F16 = 3 };

/* Widen element i of an fp32, bf16, fp16 or fp8 e4m3 array to double, exactly.  e4m3
 * (the OCP 8-bit floating-point format E4M3): sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent 0 holds the subnormals m x 2^-6 / 8; the pattern
 * with every exponent and mantissa bit set is NaN; there is no infinity. */
static double widen(const void *base, int dtype, size_t i)
{
    if (dtype == ORACLE_BF16) {   /* the upper half of a binary32 */
        uint16_t h = ((const uint16_t *)base)[i];
        uint32_t u = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
    if (dtype == ORACLE_E4M3) {
        uint8_t b = ((const uint8_t *)base)[i];
        int e = (b >> 3) & 0xF, m = b & 7;
        double v;
        if (e == 0xF && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m, -9);
        else
            v = ldexp(8.0 + m, e - 10);
        return (b & 0x80) ? -v : v;
    }
    /* ORACLE_F16, IEEE binary16: 5 exponent bits with bias 15, 10 mantissa bits */
    uint16_t b = ((const uint16_t *)base)[i];
    int e = (b >> 10) & 0x1F, m = b & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp(1024.0 + m, e - 25);
    return (b & 0x8000) ? -v : v;
}

static int clamp_n(int32_t n, int max_blocks)
{
    if (n < 0) return 0;
    if (n > max_blocks) return max_blocks;
    return (int)n;
}

/*
 * Block scores in double.  q: [nq][H][D], w: [nq][H] fp32, kblk: [max_blocks][D].
 * out: [nq][max_blocks]; entries at b >= n_blocks[q] are set to 0.
 * Returns 0, or -1 on a bad argument.
 */
int qsa_oracle_block_scores(const void *q, const float *w, const void *kblk, int dtype,
                            const int32_t *n_blocks, int nq, int n_heads, int head_dim,
                            int max_blocks, double *out)
{
    if (!q || !w || !kblk || !n_blocks || !out) return -1;
    if (nq < 0 || n_heads <= 0 || head_dim <= 0 || max_blocks < 0) return -1;
    if (dtype < ORACLE_F32 || dtype > ORACLE_F16) return -1;
    for (int qi = 0; qi < nq; ++qi) {
        int n = clamp_n(n_blocks[qi], max_blocks);
        for (int b = 0; b < max_blocks; ++b) {
            double s = 0.0;
            if (b < n) {
                for (int h = 0; h < n_heads; ++h) {
                    double dot = 0.0;
                    size_t qrow = ((size_t)qi * n_heads + h) * head_dim;
                    size_t krow = (size_t)b * head_dim;
                    for (int d = 0; d < head_dim; ++d)
                        dot += widen(q, dtype, qrow + d) * widen(kblk, dtype, krow + d);
                    double relu = dot > 0.0 ? dot : 0.0;
                    s += (double)w[(size_t)qi * n_heads + h] * relu;
                }
            }
            out[(size_t)qi * max_blocks + b] = s;
        }
    }
    return 0;
}

typedef struct {
    double score;
    int32_t id;
} scored_block;

/* Order: score descending, then id ascending. */
static int by_score_desc_id_asc(const void *pa, const void *pb)
{
    const scored_block *a = (const scored_block *)pa, *b = (const scored_block *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static int by_int_asc(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Select one query's k blocks from n scores; ids out[0..k) ascending, -1 padded. */
static int select_row(const double *row, int n, int k, int32_t *out)
{
    scored_block *list = (scored_block *)malloc((size_t)(n > 0 ? n : 1) * sizeof *list);
    if (!list) return -1;
    for (int b = 0; b < n; ++b) {
        list[b].score = row[b];
        list[b].id = b;
    }
    qsort(list, (size_t)n, sizeof *list, by_score_desc_id_asc);
    int m = n < k ? n : k;
    for (int i = 0; i < m; ++i) out[i] = list[i].id;
    qsort(out, (size_t)m, sizeof *out, by_int_asc);
    for (int i = m; i < k; ++i) out[i] = -1;
    free(list);
    return 0;
}

/*
 * Top-k over double scores [nq][stride]; ids: [nq][k].
 * n_blocks[q] is clamped to [0, max_blocks].  Returns 0, or -1 on error.
 */
int qsa_oracle_select(const double *scores, int64_t stride, const int32_t *n_blocks, int nq,
                      int max_blocks, int k, int32_t *ids)
{
    if (!scores || !n_blocks || !ids || nq < 0 || k <= 0 || stride < max_blocks) return -1;
    for (int qi = 0; qi < nq; ++qi) {
        int n = clamp_n(n_blocks[qi], max_blocks);
        if (select_row(scores + (size_t)qi * stride, n, k, ids + (size_t)qi * k)) return -1;
    }
    return 0;
}

/*
 * The same selection over fp32 scores (for instance the GPU's own), each
 * widened exactly to double before the comparison.
 */
int qsa_oracle_select_f32(const float *scores, int64_t stride, const int32_t *n_blocks, int nq,
                          int max_blocks, int k, int32_t *ids)
{
    if (!scores || !n_blocks || !ids || nq < 0 || k <= 0 || stride < max_blocks) return -1;
    double *row = (double *)malloc((size_t)(max_blocks > 0 ? max_blocks : 1) * sizeof *row);
    if (!row) return -1;
    for (int qi = 0; qi < nq; ++qi) {
        int n = clamp_n(n_blocks[qi], max_blocks);
        for (int b = 0; b < n; ++b) row[b] = (double)scores[(size_t)qi * stride + b];
        if (select_row(row, n, k, ids + (size_t)qi * k)) {
            free(row);
            return -1;
        }
    }
    free(row);
    return 0;
}

/*
 * Selection attention, forward, in double: the step that consumes the selected
 * ids, as set out in "[wave] NSA: LDS optimization for block-gather in
 * selection attention" (section "Problem": each query reads the tokens of its
 * selected blocks, T blocks of block_size tokens; strategy 1: the heads of a
 * GQA group read one copy of each block's K and V).  For query qi and attention
 * head h, whose KV head is g = h / group:
 *
 *   tokens   the set of t = 64 * b + r over the distinct ids b >= 0 of
 *            ids[qi][0..k) and 0 <= r < 64, with t < min(n_tokens[qi], capacity)
 *   logits   s_t = scale * sum_d qa[qi][h][d] * kc[g][t][d]
 *   out      o[qi][h][d] = sum_t exp(s_t - m) * vc[g][t][d] / sum_t exp(s_t - m),
 *            m = max_t s_t
 *   lse      lse[qi][h] = m + log(sum_t exp(s_t - m))
 *
 * The tokens are visited in slot order; an empty set gives o = 0 and
 * lse = -inf.  Inputs are bf16 or fp16 bit patterns (dtype), widened exactly;
 * everything after that is IEEE double.  qa: [nq][n_heads][head_dim]; kc, vc:
 * [n_kv_heads][capacity][head_dim] (token rows); ids: [nq][k];
 * out: [nq][n_heads][head_dim]; lse: [nq][n_heads].
 * Returns 0, or -1 on a bad argument.
 */
int qsa_oracle_select_attention(const uint16_t *qa, const uint16_t *kc, const uint16_t *vc, int dtype,
                                const int32_t *ids, int k, const int32_t *n_tokens, int nq,
                                int n_heads, int n_kv_heads, int head_dim, int capacity,
                                double scale, double *out, double *lse)
{
    if (!qa || !kc || !vc || !ids || !n_tokens || !out || !lse) return -1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
    if (nq < 0 || k <= 0 || n_kv_heads <= 0 || n_heads <= 0 || n_heads % n_kv_heads) return -1;
    if (head_dim <= 0 || capacity < 0) return -1;
    const int group = n_heads / n_kv_heads;
    const size_t max_tok = (size_t)k * 64;
    int32_t *tok = (int32_t *)malloc(max_tok * sizeof *tok);
    double *s = (double *)malloc(max_tok * sizeof *s);
    if (!tok || !s) {
        free(tok);
        free(s);
        return -1;
    }
    for (int qi = 0; qi < nq; ++qi) {
        const int32_t *row = ids + (size_t)qi * k;
        int ntok = n_tokens[qi] < 0 ? 0 : n_tokens[qi];
        if (ntok > capacity) ntok = capacity;
        /* the query's token set, in slot order */
        int n = 0;
        for (int j = 0; j < k; ++j) {
            const int32_t b = row[j];
            if (b < 0) continue;
            int seen = 0;
            for (int i = 0; i < j; ++i) seen |= row[i] == b;
            if (seen) continue;
            for (int r = 0; r < 64; ++r) {
                const int64_t t = (int64_t)b * 64 + r;
                if (t < ntok) tok[n++] = (int32_t)t;
            }
        }
        for (int h = 0; h < n_heads; ++h) {
            const int g = h / group;
            const size_t qrow = ((size_t)qi * n_heads + h) * head_dim;
            double *o = out + ((size_t)qi * n_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (n == 0) {
                lse[(size_t)qi * n_heads + h] = -INFINITY;
                continue;
            }
            double m = -INFINITY;
            for (int i = 0; i < n; ++i) {
                const size_t krow = ((size_t)g * capacity + tok[i]) * head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += widen(qa, dtype, qrow + d) * widen(kc, dtype, krow + d);
                s[i] = scale * dot;
                if (s[i] > m) m = s[i];
            }
            double l = 0.0;
            for (int i = 0; i < n; ++i) {
                const double e = exp(s[i] - m);
                const size_t vrow = ((size_t)g * capacity + tok[i]) * head_dim;
                l += e;
                for (int d = 0; d < head_dim; ++d) o[d] += e * widen(vc, dtype, vrow + d);
            }
            for (int d = 0; d < head_dim; ++d) o[d] /= l;
            lse[(size_t)qi * n_heads + h] = m + log(l);
        }
    }
    free(tok);
    free(s);
    return 0;
}
