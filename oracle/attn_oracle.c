/*
 * attn_oracle.c -- plain, slow fp64 CPU oracle for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (definitions from the lecture pages):
 *   - "Attention and Softmax" (CS149 Lecture 9 notes, concept 8): S = Q K^T,
 *     P = row-wise softmax(S), O = P V, with the safe softmax m = max_j x_j,
 *     f = e^{x - m}, l = sum f, softmax = f / l.
 *   - "Conclusion" of the PDC course Lecture 4 (section 4.14) and CS336
 *     Lecture 5 notes section 8.1: the scores are scaled, S = Q K^T / sqrt(d);
 *     here the scale is a runtime argument.
 *   - CS336 Lecture 5 notes section 8.3 (FlashAttention forward): the
 *     logsumexp L_i = m_i + log l_i kept per row; causal masking drops keys
 *     "in the future" of the query (key j masked for j > i).
 *   - PDC course Lecture 4, section 4.9 (the KV cache that grows during
 *     inference): with Nq < Nk the Nq queries are read as the LAST Nq
 *     positions of a sequence of Nk tokens whose keys and values are all
 *     given, so query i sits at position i + (Nk - Nq) and sees keys
 *     j <= i + (Nk - Nq).  With Nq == Nk this is the plain j > i rule.  A
 *     causal call with Nq > Nk would leave rows with no visible key and is
 *     rejected.
 *   - CS149 Lecture 9 notes concept 9 (blocked softmax): the two-block merge
 *     rule m = max(m1, m2), l = e^{m1-m} l1 + e^{m2-m} l2.
 *   - CS336 Lecture 5 notes section 8.2 (online softmax): the per-block update
 *     m' = max(m, max_block x), l' = l e^{m-m'} + sum_block e^{x-m'}.
 *
 * All arithmetic is IEEE binary64 with exp/log from the C library.  Inputs are
 * given either as binary64 or as bfloat16 bit patterns (uint16); a bfloat16
 * value is widened exactly (its 16 bits are the top half of a binary32, which
 * converts to binary64 without rounding).
 *
 * Layout of every tensor: contiguous row-major [B, H, N, d] (d innermost);
 * lse is [B, H, Nq].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ABI __attribute__((visibility("default")))

/* threads the row loops run on (1 when built without OpenMP) */
ORACLE_ABI int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- exact widening of one input element ------------------------------- */

static double widen_bf16(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* dst[i] = the binary64 value of bfloat16 bit pattern src[i] (exact) */
ORACLE_ABI void oracle_widen_bf16(const uint16_t *src, double *dst, long n)
{
    for (long i = 0; i < n; ++i)
        dst[i] = widen_bf16(src[i]);
}

/* element `idx` of an input array that is binary64 (is_bf16 == 0) or bfloat16 */
static double load_elem(const void *p, size_t idx, int is_bf16)
{
    if (is_bf16)
        return widen_bf16(((const uint16_t *)p)[idx]);
    return ((const double *)p)[idx];
}

/* ---- one row of naive attention ---------------------------------------- */

/*
 * Row i of head bh: materialise the score row S_i. (length Nk) and the
 * probability row P_i., then O_i = sum_j P_ij V_j and lse_i = m_i + ln l_i.
 * Masked keys (causal j > i + (Nk - Nq)) carry -inf and contribute e^{-inf} = 0.
 * `srow` is caller scratch of Nk doubles.
 */
static void attention_row(const void *q, const void *k, const void *v, int is_bf16,
                          long Nq, long Nk, long d, long bh, long i, int causal,
                          double scale, double *srow, double *o_row, double *lse_out)
{
    const size_t qbase = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
    const size_t kvbase = (size_t)bh * (size_t)Nk * (size_t)d;
    const long pos = i + (Nk - Nq); /* position of query i in the sequence */

    /* S_ij = scale * sum_c Q_ic K_jc, masked entries -inf */
    double m = -INFINITY;
    for (long j = 0; j < Nk; ++j) {
        if (causal && j > pos) {
            srow[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        for (long c = 0; c < d; ++c)
            dot += load_elem(q, qbase + (size_t)c, is_bf16) *
                   load_elem(k, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
        srow[j] = scale * dot;
        if (srow[j] > m)
            m = srow[j];
    }

    /* safe softmax: f_j = e^{S_ij - m}, l = sum_j f_j, P_ij = f_j / l */
    double l = 0.0;
    for (long j = 0; j < Nk; ++j) {
        srow[j] = (srow[j] == -INFINITY) ? 0.0 : exp(srow[j] - m);
        l += srow[j];
    }
    for (long j = 0; j < Nk; ++j)
        srow[j] /= l;

    /* O_i = sum_j P_ij V_j */
    for (long c = 0; c < d; ++c)
        o_row[c] = 0.0;
    for (long j = 0; j < Nk; ++j) {
        if (srow[j] == 0.0)
            continue;
        for (long c = 0; c < d; ++c)
            o_row[c] += srow[j] * load_elem(v, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
    }
    *lse_out = m + log(l);
}

/*
 * Full naive attention over all (b, h, i).  q: [B,H,Nq,d], k,v: [B,H,Nk,d],
 * o: [B,H,Nq,d] binary64, lse: [B,H,Nq] binary64.  Returns 0, or -1 on a bad
 * argument / allocation failure.
 */
ORACLE_ABI int oracle_attention(const void *q, const void *k, const void *v, int is_bf16,
                                double *o, double *lse, long B, long H, long Nq, long Nk,
                                long d, int causal, double scale)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || (causal && Nq > Nk))
        return -1;
    const long rows = B * H * Nq;
    int err = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)Nk * sizeof(double));
        if (!srow) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long r = 0; r < rows; ++r) {
                const long bh = r / Nq, i = r % Nq;
                attention_row(q, k, v, is_bf16, Nq, Nk, d, bh, i, causal, scale, srow,
                              o + (size_t)r * (size_t)d, lse + r);
            }
            free(srow);
        }
    }
    return err;
}

/*
 * The same computation restricted to a list of rows: rows[2*t] = bh (the flat
 * b*H + h index), rows[2*t+1] = i.  o: [nrows, d], lse: [nrows].  Rows are
 * independent, so a sampled row is checked exactly.
 */
ORACLE_ABI int oracle_attention_rows(const void *q, const void *k, const void *v, int is_bf16,
                                     const long *rows, long nrows, double *o, double *lse,
                                     long B, long H, long Nq, long Nk, long d, int causal,
                                     double scale)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || nrows < 0 || (causal && Nq > Nk))
        return -1;
    for (long t = 0; t < nrows; ++t)
        if (rows[2 * t] < 0 || rows[2 * t] >= B * H || rows[2 * t + 1] < 0 ||
            rows[2 * t + 1] >= Nq)
            return -1;
    int err = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)Nk * sizeof(double));
        if (!srow) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long t = 0; t < nrows; ++t)
                attention_row(q, k, v, is_bf16, Nq, Nk, d, rows[2 * t], rows[2 * t + 1], causal,
                              scale, srow, o + (size_t)t * (size_t)d, lse + t);
            free(srow);
        }
    }
    return err;
}

/* ---- online softmax, per-block form (CS336 Lecture 5 notes, 8.2) ------- */

/*
 * Process x[0..n) block by block; block b ends (exclusive) at ends[b]
 * (ends strictly increasing, last == n).  After each block the running
 * (m, l) are written to m_out[b], l_out[b]:
 *     m' = max(m, max_{j in block} x_j),  l' = l e^{m - m'} + sum_{j in block} e^{x_j - m'}
 * starting from m = -inf, l = 0.  Returns 0 or -1 on a bad block list.
 */
ORACLE_ABI int oracle_online_softmax_blocks(const double *x, long n, const long *ends,
                                            long nblocks, double *m_out, double *l_out)
{
    double m = -INFINITY, l = 0.0;
    long start = 0;
    for (long b = 0; b < nblocks; ++b) {
        const long end = ends[b];
        if (end <= start || end > n)
            return -1;
        double m_new = m;
        for (long j = start; j < end; ++j)
            if (x[j] > m_new)
                m_new = x[j];
        double s = 0.0;
        for (long j = start; j < end; ++j)
            s += exp(x[j] - m_new);
        l = (m == -INFINITY ? 0.0 : l * exp(m - m_new)) + s;
        m = m_new;
        m_out[b] = m;
        l_out[b] = l;
        start = end;
    }
    return start == n ? 0 : -1;
}

/* ---- two-block merge rule (CS149 Lecture 9 notes, concept 9) ----------- */

/*
 * Merge the softmax statistics of two blocks x1, x2 of one row:
 *   m = max(m1, m2),  l = e^{m1 - m} l1 + e^{m2 - m} l2
 * and, for attention, the two block outputs that are each normalised by
 * their own l (o_b = sum_{j in b} f_j V_j / l_b):
 *   o = (e^{m1 - m} l1 o1 + e^{m2 - m} l2 o2) / l.
 * o1, o2, o have d entries.
 */
ORACLE_ABI void oracle_softmax_merge(double m1, double l1, const double *o1, double m2,
                                     double l2, const double *o2, long d, double *m_out,
                                     double *l_out, double *o_out)
{
    const double m = m1 > m2 ? m1 : m2;
    const double a1 = (m1 == -INFINITY) ? 0.0 : exp(m1 - m);
    const double a2 = (m2 == -INFINITY) ? 0.0 : exp(m2 - m);
    const double l = a1 * l1 + a2 * l2;
    *m_out = m;
    *l_out = l;
    if (o_out)
        for (long c = 0; c < d; ++c)
            o_out[c] = (a1 * l1 * o1[c] + a2 * l2 * o2[c]) / l;
}

/* ---- FlashAttention forward, blocked (CS336 Lecture 5 notes, 8.3) ------ */

/*
 * The tiled algorithm as the notes state it, in binary64, for one head at a
 * time: for each query block Q_i (Br rows): O_i = 0, m_i = -inf, l_i = 0;
 * for each key/value block (K_j, V_j) (Bc rows):
 *     S_ij = scale Q_i K_j^T;  m_new = max(m_i, rowmax S_ij);  P_ij = e^{S_ij - m_new}
 *     l_i = e^{m_i - m_new} l_i + rowsum P_ij;  O_i = e^{m_i - m_new} O_i + P_ij V_j;  m_i = m_new
 * then O_i /= l_i and L_i = m_i + log l_i.  Causal key blocks that lie wholly
 * in the future of the query block are skipped; inside a block, masked keys
 * carry -inf.  Block sizes need not divide N.  Inputs binary64 only.
 * Returns 0 or -1.
 */
ORACLE_ABI int oracle_attention_blocked(const double *q, const double *k, const double *v,
                                        double *o, double *lse, long B, long H, long Nq,
                                        long Nk, long d, int causal, double scale, long Br,
                                        long Bc)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || Br <= 0 || Bc <= 0 ||
        (causal && Nq > Nk))
        return -1;
    const long off = Nk - Nq; /* query i sits at position i + off */
    double *S = (double *)malloc((size_t)Br * (size_t)Bc * sizeof(double));
    double *m = (double *)malloc((size_t)Br * sizeof(double));
    double *l = (double *)malloc((size_t)Br * sizeof(double));
    double *acc = (double *)malloc((size_t)Br * (size_t)d * sizeof(double));
    if (!S || !m || !l || !acc) {
        free(S); free(m); free(l); free(acc);
        return -1;
    }
    for (long bh = 0; bh < B * H; ++bh) {
        const double *qh = q + (size_t)bh * Nq * d;
        const double *kh = k + (size_t)bh * Nk * d;
        const double *vh = v + (size_t)bh * Nk * d;
        for (long i0 = 0; i0 < Nq; i0 += Br) {
            const long br = (i0 + Br <= Nq) ? Br : Nq - i0;
            for (long r = 0; r < br; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (long c = 0; c < d; ++c)
                    acc[r * d + c] = 0.0;
            }
            for (long j0 = 0; j0 < Nk; j0 += Bc) {
                if (causal && j0 > i0 + br - 1 + off)
                    break; /* every key of this block is after every query row */
                const long bc = (j0 + Bc <= Nk) ? Bc : Nk - j0;
                for (long r = 0; r < br; ++r) {
                    const long i = i0 + r;
                    double rowmax = -INFINITY;
                    for (long t = 0; t < bc; ++t) {
                        const long j = j0 + t;
                        double s = -INFINITY;
                        if (!(causal && j > i + off)) {
                            double dot = 0.0;
                            for (long c = 0; c < d; ++c)
                                dot += qh[i * d + c] * kh[j * d + c];
                            s = scale * dot;
                        }
                        S[r * Bc + t] = s;
                        if (s > rowmax)
                            rowmax = s;
                    }
                    const double m_new = m[r] > rowmax ? m[r] : rowmax;
                    if (m_new == -INFINITY)
                        continue; /* nothing visible yet in this row */
                    const double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                    double rowsum = 0.0;
                    for (long t = 0; t < bc; ++t) {
                        const double p = (S[r * Bc + t] == -INFINITY) ? 0.0 : exp(S[r * Bc + t] - m_new);
                        S[r * Bc + t] = p;
                        rowsum += p;
                    }
                    l[r] = alpha * l[r] + rowsum;
                    for (long c = 0; c < d; ++c) {
                        double pv = 0.0;
                        for (long t = 0; t < bc; ++t)
                            pv += S[r * Bc + t] * vh[(j0 + t) * d + c];
                        acc[r * d + c] = alpha * acc[r * d + c] + pv;
                    }
                    m[r] = m_new;
                }
            }
            for (long r = 0; r < br; ++r) {
                const size_t row = (size_t)bh * Nq + (size_t)(i0 + r);
                for (long c = 0; c < d; ++c)
                    o[row * d + c] = acc[r * d + c] / l[r];
                lse[row] = m[r] + log(l[r]);
            }
        }
    }
    free(S); free(m); free(l); free(acc);
    return 0;
}

/* ---- FlashAttention backward (CS336 Lecture 5 notes, section 8.4) ------ */

/*
 * Gradients of O = softmax(S) V with S = scale Q K^T (masked as in the
 * forward), for a given upstream gradient dO = dL/dO:
 *     P_ij  = softmax_j(S_i.)             dV_j = sum_i P_ij dO_i
 *     dP_ij = dO_i . V_j                  D_i  = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)          dQ_i = scale sum_j dS_ij K_j
 *                                         dK_j = scale sum_i dS_ij Q_i
 * D_i is written from its definition (the derivative of the softmax), not
 * from the shortcut rowsum(dO_i * O_i) the notes prove equal in exercise 9,
 * so the tests can check that identity against it.  Inputs q, k, v, dout as
 * in the forward (binary64 or bfloat16 bits), dout: [B,H,Nq,d].  Outputs are
 * binary64.
 */

/*
 * Row i of head bh: P_i. (normalised, masked entries 0) into prow, dP_i. into
 * dprow (Nk entries each, dP of masked keys left 0), D_i into *D_out, lse_i
 * into *lse_out.  `o_row` is caller scratch of d doubles.
 */
static void backward_row(const void *q, const void *k, const void *v, const void *dout,
                         int is_bf16, long Nq, long Nk, long d, long bh, long i, int causal,
                         double scale, double *prow, double *dprow, double *o_row,
                         double *D_out, double *lse_out)
{
    attention_row(q, k, v, is_bf16, Nq, Nk, d, bh, i, causal, scale, prow, o_row, lse_out);
    const size_t dobase = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
    const size_t kvbase = (size_t)bh * (size_t)Nk * (size_t)d;
    double D = 0.0;
    for (long j = 0; j < Nk; ++j) {
        dprow[j] = 0.0;
        if (prow[j] == 0.0)
            continue; /* masked (or underflowed): contributes nothing */
        double dp = 0.0;
        for (long c = 0; c < d; ++c)
            dp += load_elem(dout, dobase + (size_t)c, is_bf16) *
                  load_elem(v, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
        dprow[j] = dp;
        D += prow[j] * dp;
    }
    *D_out = D;
}

/*
 * Full backward over all heads.  dq: [B,H,Nq,d], dk, dv: [B,H,Nk,d].
 * Heads run in parallel; inside a head the rows run in order, so the result
 * does not depend on the thread count.  Returns 0 or -1.
 */
ORACLE_ABI int oracle_attention_bwd(const void *q, const void *k, const void *v,
                                    const void *dout, int is_bf16, double *dq, double *dk,
                                    double *dv, long B, long H, long Nq, long Nk, long d,
                                    int causal, double scale)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || (causal && Nq > Nk))
        return -1;
    int err = 0;
#pragma omp parallel
    {
        double *prow = (double *)malloc((size_t)Nk * sizeof(double));
        double *dprow = (double *)malloc((size_t)Nk * sizeof(double));
        double *o_row = (double *)malloc((size_t)d * sizeof(double));
        if (!prow || !dprow || !o_row) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bh = 0; bh < B * H; ++bh) {
                double *dkh = dk + (size_t)bh * (size_t)Nk * (size_t)d;
                double *dvh = dv + (size_t)bh * (size_t)Nk * (size_t)d;
                for (size_t x = 0; x < (size_t)Nk * (size_t)d; ++x) {
                    dkh[x] = 0.0;
                    dvh[x] = 0.0;
                }
                const size_t kvbase = (size_t)bh * (size_t)Nk * (size_t)d;
                for (long i = 0; i < Nq; ++i) {
                    double D, lse;
                    backward_row(q, k, v, dout, is_bf16, Nq, Nk, d, bh, i, causal, scale, prow,
                                 dprow, o_row, &D, &lse);
                    const size_t rbase = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
                    double *dqi = dq + rbase;
                    for (long c = 0; c < d; ++c)
                        dqi[c] = 0.0;
                    for (long j = 0; j < Nk; ++j) {
                        const double p = prow[j];
                        if (p == 0.0)
                            continue;
                        const double ds = p * (dprow[j] - D);
                        for (long c = 0; c < d; ++c) {
                            const double kjc = load_elem(k, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
                            const double qic = load_elem(q, rbase + (size_t)c, is_bf16);
                            const double doic = load_elem(dout, rbase + (size_t)c, is_bf16);
                            dqi[c] += scale * ds * kjc;
                            dkh[(size_t)j * (size_t)d + (size_t)c] += scale * ds * qic;
                            dvh[(size_t)j * (size_t)d + (size_t)c] += p * doic;
                        }
                    }
                }
            }
        }
        free(prow);
        free(dprow);
        free(o_row);
    }
    return err;
}

/*
 * dQ on a list of rows (rows[2t] = bh, rows[2t+1] = i); dq: [nrows, d].
 * Optionally the per-row D_i (D may be NULL), for the exercise-9 check.
 */
ORACLE_ABI int oracle_attention_bwd_dq_rows(const void *q, const void *k, const void *v,
                                            const void *dout, int is_bf16, const long *rows,
                                            long nrows, double *dq, double *D, long B, long H,
                                            long Nq, long Nk, long d, int causal, double scale)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || nrows < 0 || (causal && Nq > Nk))
        return -1;
    for (long t = 0; t < nrows; ++t)
        if (rows[2 * t] < 0 || rows[2 * t] >= B * H || rows[2 * t + 1] < 0 ||
            rows[2 * t + 1] >= Nq)
            return -1;
    int err = 0;
#pragma omp parallel
    {
        double *prow = (double *)malloc((size_t)Nk * sizeof(double));
        double *dprow = (double *)malloc((size_t)Nk * sizeof(double));
        double *o_row = (double *)malloc((size_t)d * sizeof(double));
        if (!prow || !dprow || !o_row) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long t = 0; t < nrows; ++t) {
                const long bh = rows[2 * t], i = rows[2 * t + 1];
                double Di, lse;
                backward_row(q, k, v, dout, is_bf16, Nq, Nk, d, bh, i, causal, scale, prow,
                             dprow, o_row, &Di, &lse);
                if (D)
                    D[t] = Di;
                const size_t kvbase = (size_t)bh * (size_t)Nk * (size_t)d;
                double *dqi = dq + (size_t)t * (size_t)d;
                for (long c = 0; c < d; ++c)
                    dqi[c] = 0.0;
                for (long j = 0; j < Nk; ++j) {
                    if (prow[j] == 0.0)
                        continue;
                    const double ds = prow[j] * (dprow[j] - Di);
                    for (long c = 0; c < d; ++c)
                        dqi[c] += scale * ds * load_elem(k, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
                }
            }
        }
        free(prow);
        free(dprow);
        free(o_row);
    }
    return err;
}

/*
 * dK and dV on a list of keys (keys[2t] = bh, keys[2t+1] = j); dk, dv:
 * [nkeys, d].  For each head that appears, every row's lse_i and D_i are
 * computed first (rows in parallel); then each listed key sums over the rows
 * with P_ij = e^{S_ij - lse_i} recomputed from the logsumexp, the form the
 * notes use in the backward pass (section 8.4).  Returns 0 or -1.
 */
ORACLE_ABI int oracle_attention_bwd_dkdv_keys(const void *q, const void *k, const void *v,
                                              const void *dout, int is_bf16, const long *keys,
                                              long nkeys, double *dk, double *dv, long B,
                                              long H, long Nq, long Nk, long d, int causal,
                                              double scale)
{
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || nkeys < 0 || (causal && Nq > Nk))
        return -1;
    for (long t = 0; t < nkeys; ++t)
        if (keys[2 * t] < 0 || keys[2 * t] >= B * H || keys[2 * t + 1] < 0 ||
            keys[2 * t + 1] >= Nk)
            return -1;
    double *lse = (double *)malloc((size_t)Nq * sizeof(double));
    double *Dr = (double *)malloc((size_t)Nq * sizeof(double));
    char *done = (char *)calloc((size_t)(nkeys > 0 ? nkeys : 1), 1);
    if (!lse || !Dr || !done) {
        free(lse); free(Dr); free(done);
        return -1;
    }
    int err = 0;
    for (long t0 = 0; t0 < nkeys && !err; ++t0) {
        if (done[t0])
            continue;
        const long bh = keys[2 * t0];
        /* pass 1: lse_i and D_i of every row of this head */
#pragma omp parallel
        {
            double *prow = (double *)malloc((size_t)Nk * sizeof(double));
            double *dprow = (double *)malloc((size_t)Nk * sizeof(double));
            double *o_row = (double *)malloc((size_t)d * sizeof(double));
            if (!prow || !dprow || !o_row) {
#pragma omp atomic write
                err = -1;
            } else {
#pragma omp for schedule(dynamic, 8)
                for (long i = 0; i < Nq; ++i)
                    backward_row(q, k, v, dout, is_bf16, Nq, Nk, d, bh, i, causal, scale, prow,
                                 dprow, o_row, &Dr[i], &lse[i]);
            }
            free(prow);
            free(dprow);
            free(o_row);
        }
        if (err)
            break;
        /* pass 2: every listed key of this head */
        const size_t kvbase = (size_t)bh * (size_t)Nk * (size_t)d;
        const size_t qbase = (size_t)bh * (size_t)Nq * (size_t)d;
#pragma omp parallel for schedule(dynamic, 1)
        for (long t = t0; t < nkeys; ++t) {
            if (keys[2 * t] != bh)
                continue;
            done[t] = 1;
            const long j = keys[2 * t + 1];
            double *dkj = dk + (size_t)t * (size_t)d;
            double *dvj = dv + (size_t)t * (size_t)d;
            for (long c = 0; c < d; ++c) {
                dkj[c] = 0.0;
                dvj[c] = 0.0;
            }
            for (long i = 0; i < Nq; ++i) {
                if (causal && j > i + (Nk - Nq))
                    continue;
                double s = 0.0, dp = 0.0;
                for (long c = 0; c < d; ++c) {
                    const double vjc = load_elem(v, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
                    s += load_elem(q, qbase + (size_t)i * (size_t)d + (size_t)c, is_bf16) *
                         load_elem(k, kvbase + (size_t)j * (size_t)d + (size_t)c, is_bf16);
                    dp += load_elem(dout, qbase + (size_t)i * (size_t)d + (size_t)c, is_bf16) * vjc;
                }
                const double p = exp(scale * s - lse[i]);
                const double ds = p * (dp - Dr[i]);
                for (long c = 0; c < d; ++c) {
                    dkj[c] += scale * ds * load_elem(q, qbase + (size_t)i * (size_t)d + (size_t)c, is_bf16);
                    dvj[c] += p * load_elem(dout, qbase + (size_t)i * (size_t)d + (size_t)c, is_bf16);
                }
            }
        }
    }
    free(lse);
    free(Dr);
    free(done);
    return err;
}

/* ---- FP8 (E4M3) inputs --------------------------------------------------- */

/*
 * Value of one 8-bit E4M3 code, the FP8 number format the lecture pages name
 * for Blackwell's low-precision tensor cores (CS336 Lecture 5 notes, section
 * 6.2; PDC course Lecture 7, section 7.14).  The pages name the format without
 * spelling out its bits; the definition followed here is the OCP 8-bit floating
 * point specification's E4M3: bit 7 the sign, bits 6-3 a biased exponent
 * (bias 7), bits 2-0 the mantissa; exponent field 0 holds the subnormals
 * (mantissa / 8) * 2^(1 - 7); the code with every exponent and mantissa bit
 * set is NaN; there is no infinity, so the largest finite value is
 * (1 + 6/8) * 2^8 = 448.
 */
static double e4m3_value(uint8_t code)
{
    const int sign = (code >> 7) & 1;
    const int e = (code >> 3) & 15;
    const int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * dst[i] = descale * value(src[i]) for n codes: the per-tensor dequantisation
 * of an FP8 operand (PDC course Lecture 7, section 7.14: one scale per
 * tensor).  The product of a 4-bit significand and a binary32 descale is
 * exact in binary64.
 */
ORACLE_ABI void oracle_decode_e4m3(const uint8_t *src, double *dst, long n, double descale)
{
    for (long i = 0; i < n; ++i)
        dst[i] = descale * e4m3_value(src[i]);
}

/* ---- MX (microscaling) FP8 inputs --------------------------------------- */

/*
 * Value of one E8M0 block-scale code.  PDC course Lecture 7, section 7.14
 * names the MX ("microscaling") formats for fine-grained quantisation on
 * Blackwell without spelling out their bits; the definition followed here is
 * the OCP Microscaling Formats (MX) v1.0 specification's E8M0: an unsigned
 * 8-bit exponent with bias 127, value 2^(code - 127), no sign and no mantissa;
 * the code 0xFF is NaN.
 */
static double e8m0_value(uint8_t code)
{
    if (code == 0xFF)
        return NAN;
    return ldexp(1.0, (int)code - 127);
}

/*
 * MXFP8 dequantisation (same specification): `rows` rows of `d` E4M3 codes,
 * the elements c of a row in blocks of `block` consecutive ones (32 for the
 * MX formats), block b of row r sharing the scale scales[r * (d / block) + b]:
 *   dst[r * d + c] = E8M0(scales[r * nb + c / block]) * E4M3(codes[r * d + c]).
 * Returns 0, or -1 when d is not a multiple of block.
 */
ORACLE_ABI int oracle_decode_mx(const uint8_t *codes, const uint8_t *scales, double *dst,
                                long rows, long d, long block)
{
    if (block <= 0 || d % block != 0)
        return -1;
    const long nb = d / block;
    for (long r = 0; r < rows; ++r)
        for (long c = 0; c < d; ++c)
            dst[r * d + c] = e8m0_value(scales[r * nb + c / block]) * e4m3_value(codes[r * d + c]);
    return 0;
}
