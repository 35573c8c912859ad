/*
 * attn_oracle.c -- plain fp64 CPU reference for exact scaled-dot-product
 * attention, its logsumexp, and the log-sum-exp merge of partial results.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this code.  It shares nothing with
 * the CUDA path: no headers, no helpers, no constants.
 *
 * What it computes (the "standard attention" of the lecture notes
 * "Optimizing Attention for Modern Hardware: FlashAttention 1-4",
 * sections 0.4 and 1.4, and of the blog "FlashAttention: tiling + recomputation",
 * section 1.1):
 *
 *   for every (b, hq, i), with kv head g = hq / (Hq / Hkv)       (reading: GQA
 *                                                                 groups are
 *                                                                 contiguous)
 *     s_ij  = scale * sum_c q[b,hq,i,c] * k[b,g,j,c]            for allowed j
 *     LSE_i = log sum_j exp(s_ij)                                natural log
 *     O_i   = sum_j exp(s_ij - LSE_i) * v[b,g,j,:]
 *
 *   allowed j:  window_lo <= j < window_hi        (a key window; default all)
 *               j < kv_len[b]                      (decode: valid KV prefix)
 *               j <= i + (Nk - Nq)   if causal     (reading: bottom-right
 *                                                   alignment; equals j <= i
 *                                                   when Nq == Nk, notes 2.5)
 *   a row with no allowed key gets O = 0 and LSE = -inf (reading: the pages
 *   never reach this case).
 *
 * It is the three-kernel "Algorithm 0" done one query row at a time: pass 1
 * forms the score row S_i, pass 2 takes the max-subtracted softmax of it, pass
 * 3 multiplies the probabilities into V.  Rows are independent, so working row
 * by row is still the plain definition and bounds memory at O(Nk).
 *
 * The merge (notes section 6.1, exercise 3) combines partial results (LSE_s,
 * O_s) of disjoint key sets: M = max_s LSE_s, w_s = exp(LSE_s - M),
 * O = sum_s w_s O_s / sum_s w_s, LSE = M + log sum_s w_s.
 *
 * The gradients (lecture notes section 2.6; "FlashAttention: tiling +
 * recomputation", section 3.3) for an upstream gradient dO of O, per row i
 * with P_ij = exp(s_ij - LSE_i) over the allowed keys:
 *
 *   dP_ij = dO_i . v_j                 D_i  = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)         (the softmax Jacobian applied to dP)
 *   dQ_i  = scale sum_j dS_ij k_j      dK_j = scale sum_i dS_ij q_i
 *   dV_j  = sum_i P_ij dO_i
 *
 * summed over the query heads of a KV head's group for dK and dV.  D is taken
 * from its definition here (the kernels use the identity D_i = dO_i . O_i).
 *
 * Inputs are bf16 bit patterns (uint16); widening bf16 to double is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row: the three passes over its score row.  s_row is scratch of
 * length Nk.  Returns nothing; writes d values to o_row and one to *lse. */
static void attention_row(const uint16_t *q_row, const uint16_t *k_head,
                          const uint16_t *v_head, int Nk, int d, double scale,
                          int j_begin, int j_end, double *s_row, double *q_dbl,
                          double *o_row, double *lse) {
    int j, c;
    for (c = 0; c < d; ++c) {
        q_dbl[c] = bf16_bits_to_double(q_row[c]);
        o_row[c] = 0.0;
    }
    if (j_end <= j_begin) {
        *lse = -INFINITY;
        return;
    }
    /* pass 1: scores */
    for (j = j_begin; j < j_end; ++j) {
        const uint16_t *k_row = k_head + (size_t)j * d;
        double acc = 0.0;
        for (c = 0; c < d; ++c) acc += q_dbl[c] * bf16_bits_to_double(k_row[c]);
        s_row[j] = scale * acc;
    }
    /* pass 2: max-subtracted softmax numerators and their sum */
    double m = -INFINITY;
    for (j = j_begin; j < j_end; ++j)
        if (s_row[j] > m) m = s_row[j];
    double l = 0.0;
    for (j = j_begin; j < j_end; ++j) {
        s_row[j] = exp(s_row[j] - m);
        l += s_row[j];
    }
    /* pass 3: probabilities times V */
    for (j = j_begin; j < j_end; ++j) {
        const uint16_t *v_row = v_head + (size_t)j * d;
        double p = s_row[j] / l;
        for (c = 0; c < d; ++c) o_row[c] += p * bf16_bits_to_double(v_row[c]);
    }
    *lse = m + log(l);
    (void)Nk;
}

/*
 * Attention for an explicit list of query rows.
 *   q: [B, Hq, Nq, d]  k, v: [B, Hkv, Nk, d]   (bf16 bits, row-major)
 *   kv_len: NULL or [B] valid key counts
 *   window_lo, window_hi: key window; window_hi <= 0 means Nk
 *   rows: n_rows triples (b, hq, i)
 *   o_out: [n_rows, d]   lse_out: [n_rows]
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int B, int Hq, int Hkv, int Nq, int Nk, int d,
                          int causal, double scale, const int32_t *kv_len,
                          int window_lo, int window_hi,
                          long n_rows, const int32_t *rows,
                          double *o_out, double *lse_out, int n_threads) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (Hq % Hkv != 0) return -1;
    if (window_hi <= 0 || window_hi > Nk) window_hi = Nk;
    if (window_lo < 0) window_lo = 0;
    const int group = Hq / Hkv;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel
    {
        double *s_row = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *q_dbl = (double *)malloc(sizeof(double) * (size_t)d);
        long r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            int b = rows[3 * r], hq = rows[3 * r + 1], i = rows[3 * r + 2];
            if (b < 0 || b >= B || hq < 0 || hq >= Hq || i < 0 || i >= Nq) {
                bad = 1;
                continue;
            }
            int g = hq / group;
            int j_begin = window_lo;
            int j_end = window_hi;
            if (kv_len && kv_len[b] < j_end) j_end = kv_len[b];
            if (causal) {
                long last = (long)i + (long)(Nk - Nq); /* last allowed key */
                if (last + 1 < j_end) j_end = (int)(last + 1 < 0 ? 0 : last + 1);
            }
            const uint16_t *q_row = q + (((size_t)b * Hq + hq) * Nq + i) * d;
            const uint16_t *k_head = k + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            const uint16_t *v_head = v + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            attention_row(q_row, k_head, v_head, Nk, d, scale, j_begin, j_end,
                          s_row, q_dbl, o_out + (size_t)r * d, lse_out + r);
        }
        free(s_row);
        free(q_dbl);
    }
    return bad ? -1 : 0;
}

/* Every row, in [B, Hq, Nq] order: o_out [B, Hq, Nq, d], lse_out [B, Hq, Nq]. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     double scale, const int32_t *kv_len, int window_lo,
                     int window_hi, double *o_out, double *lse_out, int n_threads) {
    if (B < 1 || Hq < 1 || Nq < 1) return -1;
    long n_rows = (long)B * Hq * Nq;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * 3 * (size_t)n_rows);
    if (!rows) return -1;
    long r = 0;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h)
            for (int i = 0; i < Nq; ++i) {
                rows[3 * r] = b;
                rows[3 * r + 1] = h;
                rows[3 * r + 2] = i;
                ++r;
            }
    int rc = oracle_attention_rows(q, k, v, B, Hq, Hkv, Nq, Nk, d, causal, scale,
                                   kv_len, window_lo, window_hi, n_rows, rows,
                                   o_out, lse_out, n_threads);
    free(rows);
    return rc;
}

/*
 * Log-sum-exp merge of n partial results over disjoint key sets.
 *   lse_parts: [n]   o_parts: [n, d] (each already normalised by its own sum)
 * Writes lse_out[0] and o_out[0..d).  Parts with LSE = -inf carry no weight.
 */
void oracle_lse_merge(int n, int d, const double *lse_parts, const double *o_parts,
                      double *lse_out, double *o_out) {
    int s, c;
    double M = -INFINITY;
    for (s = 0; s < n; ++s)
        if (lse_parts[s] > M) M = lse_parts[s];
    for (c = 0; c < d; ++c) o_out[c] = 0.0;
    if (M == -INFINITY) {
        *lse_out = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (s = 0; s < n; ++s) {
        double w = exp(lse_parts[s] - M);
        wsum += w;
        for (c = 0; c < d; ++c) o_out[c] += w * o_parts[(size_t)s * d + c];
    }
    for (c = 0; c < d; ++c) o_out[c] /= wsum;
    *lse_out = M + log(wsum);
}

/*
 * Gradients of every row (see the header).  dout is bf16 like q, k, v;
 * dq_out [B, Hq, Nq, d], dk_out and dv_out [B, Hkv, Nk, d].  One task per
 * (b, KV head), so the sums over a group's query heads need no locks.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int B, int Hq, int Hkv, int Nq, int Nk,
                         int d, int causal, double scale, double *dq_out,
                         double *dk_out, double *dv_out, int n_threads) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (Hq % Hkv != 0) return -1;
    const int group = Hq / Hkv;
    const long n_groups = (long)B * Hkv;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    memset(dq_out, 0, sizeof(double) * (size_t)B * Hq * Nq * d);
    memset(dk_out, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    memset(dv_out, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);

#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *qi = (double *)malloc(sizeof(double) * (size_t)d);
        double *doi = (double *)malloc(sizeof(double) * (size_t)d);
        long t;
#pragma omp for schedule(dynamic, 1)
        for (t = 0; t < n_groups; ++t) {
            const int b = (int)(t / Hkv), g = (int)(t % Hkv);
            const uint16_t *kh = k + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            const uint16_t *vh = v + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            double *dkh = dk_out + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            double *dvh = dv_out + ((size_t)b * Hkv + g) * (size_t)Nk * d;
            for (int hq = g * group; hq < (g + 1) * group; ++hq) {
                for (int i = 0; i < Nq; ++i) {
                    const size_t row = ((size_t)b * Hq + hq) * Nq + i;
                    int j_end = Nk;
                    if (causal) {
                        long last = (long)i + (long)(Nk - Nq);
                        if (last + 1 < j_end) j_end = (int)(last + 1 < 0 ? 0 : last + 1);
                    }
                    if (j_end <= 0) continue; /* no allowed key: all gradients 0 */
                    for (int c = 0; c < d; ++c) {
                        qi[c] = bf16_bits_to_double(q[row * d + c]);
                        doi[c] = bf16_bits_to_double(dout[row * d + c]);
                    }
                    /* P_i: the softmax of the scaled scores over the allowed keys */
                    double m = -INFINITY;
                    for (int j = 0; j < j_end; ++j) {
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c)
                            acc += qi[c] * bf16_bits_to_double(kh[(size_t)j * d + c]);
                        p[j] = scale * acc;
                        if (p[j] > m) m = p[j];
                    }
                    double sum = 0.0;
                    for (int j = 0; j < j_end; ++j) {
                        p[j] = exp(p[j] - m);
                        sum += p[j];
                    }
                    for (int j = 0; j < j_end; ++j) p[j] /= sum;
                    /* dP_i = dO_i V^T and D_i = sum_j P_ij dP_ij */
                    double D = 0.0;
                    for (int j = 0; j < j_end; ++j) {
                        double acc = 0.0;
                        for (int c = 0; c < d; ++c)
                            acc += doi[c] * bf16_bits_to_double(vh[(size_t)j * d + c]);
                        dp[j] = acc;
                        D += p[j] * acc;
                    }
                    /* dS, then the three products */
                    double *dqi = dq_out + row * d;
                    for (int j = 0; j < j_end; ++j) {
                        const double ds = p[j] * (dp[j] - D);
                        for (int c = 0; c < d; ++c) {
                            dqi[c] += scale * ds * bf16_bits_to_double(kh[(size_t)j * d + c]);
                            dkh[(size_t)j * d + c] += scale * ds * qi[c];
                            dvh[(size_t)j * d + c] += p[j] * doi[c];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
        free(qi);
        free(doi);
    }
    return 0;
}
