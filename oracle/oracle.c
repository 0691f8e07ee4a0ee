/*
 * Exact-attention oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. This file is the checker for the CUDA path, not part of
 * it: only the tests, the package's smoke check and the CPU-baseline leg of the
 * benchmark load it. It shares no code, header, table or helper with the CUDA
 * library, and the product never calls it.
 *
 * What it computes is the textbook definition, written out with no blocking,
 * fusion or online recurrence:
 *
 *   S = scale * Q K^T + B          ("Understanding FlashAttention Pt 1", §0.2
 *                                    Notation; bias added after scaling)
 *   P = row-softmax(S), O = P V    (same section)
 *
 * with the safe (max-subtracted) two-pass softmax of "Understanding
 * FlashAttention Pt 1" §2.2 and "FlashAttention, Explained" §9: first the row
 * maximum m, then l = sum_j exp(s_j - m), then p_j = exp(s_j - m) / l.
 * Every query row is materialised in full (all Nk scores) before any of it is
 * used. The saved statistic is the natural-log log-sum-exp
 * LSE_i = m_i + ln(l_i) ("flash-attention", Part VI: its worked example adds
 * the natural log of the final denominator to the final max).
 *
 * Masking:
 *  - key-padding bias: bias[b][j] is added to every score of key j in batch b;
 *    -inf means "masked" ("Understanding FlashAttention Pt 1", §3.5: masked
 *    entries get -inf before the softmax and so probability 0);
 *  - causal: key j is allowed for query i iff j <= i + (Nk - Nq), i.e. the
 *    bottom-right alignment described in "flash-attention" (causal
 *    cross-attention shapes); for Nq == Nk this is the plain lower triangle
 *    of "Understanding FlashAttention Pt 1" §3.5.
 *  - a row whose every score is -inf gets O = 0 and LSE = -inf
 *    ("flash-attention", Part VI: a fully masked row produces zeros, not NaN;
 *    LSE = log of an empty sum = -inf is this library's reading).
 *
 * The backward is the softmax Jacobian written out per row
 * ("FlashAttention: Mathematical Foundations...", §4 backward;
 * "FlashAttention, Explained", §17):
 *   dV = P^T dO,  dP = dO V^T,
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)     <- computed from P and dP,
 *                                                  NOT via rowsum(dO o O), so
 *                                                  the tests can check that
 *                                                  identity instead of assuming it
 *   dQ = scale * dS K,  dK = scale * dS^T Q.
 * Masked entries have P = 0 and so dS = 0. No gradient flows to the bias.
 *
 * Layout: every tensor is contiguous [B][H][N][d] (d innermost), bias is
 * [B][Nk]. All arithmetic is double; sums run in plain index order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int key_allowed(int i, int j, int Nq, int Nk, int causal)
{
    if (!causal) return 1;
    return (long)j <= (long)i + (long)Nk - (long)Nq;
}

/* Score row s[0..Nk) of query i of one head; returns the row maximum. */
static double score_row(const double *qi, const double *kh, const double *bias_b,
                        int i, int Nq, int Nk, int d, double scale, int causal,
                        double *s)
{
    double m = -INFINITY;
    for (int j = 0; j < Nk; ++j) {
        double v;
        if (!key_allowed(i, j, Nq, Nk, causal)) {
            v = -INFINITY;
        } else {
            const double *kj = kh + (size_t)j * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qi[c] * kj[c];
            v = scale * dot;
            if (bias_b) v += bias_b[j];   /* -inf stays -inf */
        }
        s[j] = v;
        if (v > m) m = v;
    }
    return m;
}

/* Two-pass safe softmax of a materialised row, in place: s -> p.
 * Returns LSE (natural log); -inf and p == 0 for a fully masked row. */
static double softmax_row(double *s, int Nk, double m)
{
    if (m == -INFINITY) {
        for (int j = 0; j < Nk; ++j) s[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int j = 0; j < Nk; ++j) l += exp(s[j] - m);   /* exp(-inf) == 0 */
    for (int j = 0; j < Nk; ++j) s[j] = exp(s[j] - m) / l;
    return m + log(l);
}

/*
 * Forward of one head for a list of query rows: rows[r] when rows != NULL,
 * else row0 + r, for r in [0, nrows).
 * q [Nq][d], k,v [Nk][d], bias [Nk] or NULL; o [nrows][d], lse [nrows] are
 * written in that order.
 */
static void fwd_head_rows(const double *q, const double *k, const double *v,
                          const double *bias, const int *rows, int row0, int nrows,
                          double *o, double *lse, int Nq, int Nk, int d,
                          double scale, int causal, double *s)
{
    for (int r = 0; r < nrows; ++r) {
        int i = rows ? rows[r] : row0 + r;
        const double *qi = q + (size_t)i * d;
        double m = score_row(qi, k, bias, i, Nq, Nk, d, scale, causal, s);
        double L = softmax_row(s, Nk, m);
        double *oi = o + (size_t)r * d;
        for (int c = 0; c < d; ++c) oi[c] = 0.0;
        for (int j = 0; j < Nk; ++j) {
            double p = s[j];
            if (p == 0.0) continue;   /* zero weight; also keeps masked NaN rows of V out */
            const double *vj = v + (size_t)j * d;
            for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
        }
        lse[r] = L;
    }
}

/*
 * Full forward. Parallel over (b, h, row chunks); each thread holds one
 * materialised score row of Nk doubles at a time.
 * Returns 0, or -1 if scratch could not be allocated.
 */
int oracle_fwd(const double *q, const double *k, const double *v,
               const double *bias, double *o, double *lse,
               int B, int H, int Nq, int Nk, int d, double scale, int causal)
{
    const long BH = (long)B * H;
    const int CH = 64;                       /* rows per task */
    const long nch = (Nq + CH - 1) / CH;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < BH * nch; ++t) {
            if (!s) continue;
            long bh = t / nch, c = t % nch;
            int b = (int)(bh / H);
            int r0 = (int)(c * CH), r1 = r0 + CH < Nq ? r0 + CH : Nq;
            size_t qoff = (size_t)bh * Nq * d, koff = (size_t)bh * Nk * d;
            fwd_head_rows(q + qoff, k + koff, v + koff,
                          bias ? bias + (size_t)b * Nk : NULL, NULL, r0, r1 - r0,
                          o + qoff + (size_t)r0 * d, lse + (size_t)bh * Nq + r0,
                          Nq, Nk, d, scale, causal, s);
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * Forward for selected rows of selected heads: for t in [0, n), head
 * bh = heads[t] (flat b*H + h) and query row rows[t]. o [n][d], lse [n].
 */
int oracle_fwd_rows(const double *q, const double *k, const double *v,
                    const double *bias, const long *heads, const int *rows,
                    long n, double *o, double *lse,
                    int B, int H, int Nq, int Nk, int d, double scale, int causal)
{
    (void)B;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < n; ++t) {
            if (!s) continue;
            long bh = heads[t];
            int b = (int)(bh / H);
            size_t qoff = (size_t)bh * Nq * d, koff = (size_t)bh * Nk * d;
            fwd_head_rows(q + qoff, k + koff, v + koff,
                          bias ? bias + (size_t)b * Nk : NULL, rows + t, 0, 1,
                          o + (size_t)t * d, lse + t, Nq, Nk, d, scale, causal, s);
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * Backward of one head, row by row: each query row's S, P and dP are
 * materialised in full, then its dS row is formed from the Jacobian and
 * scattered into dQ (row i), dK and dV (all keys).
 * dq [Nq][d] is written; dk, dv [Nk][d] must be zeroed by the caller.
 * If rows != NULL only those query rows are processed: dq [nrows][d] is
 * written in the order of rows, and, when dk and dv are not NULL, the
 * contributions of exactly those rows are added into them.
 */
static void bwd_head(const double *q, const double *k, const double *v,
                     const double *bias, const double *dO,
                     double *dq, double *dk, double *dv,
                     const int *rows, int nrows,
                     int Nq, int Nk, int d, double scale, int causal,
                     double *p, double *dp)
{
    for (int r = 0; r < nrows; ++r) {
        int i = rows ? rows[r] : r;
        const double *qi = q + (size_t)i * d;
        const double *doi = dO + (size_t)i * d;
        double m = score_row(qi, k, bias, i, Nq, Nk, d, scale, causal, p);
        softmax_row(p, Nk, m);
        /* dP_ij = dO_i . V_j ; rowdot = sum_j P_ij dP_ij */
        double rowdot = 0.0;
        for (int j = 0; j < Nk; ++j) {
            if (p[j] == 0.0) { dp[j] = 0.0; continue; }
            const double *vj = v + (size_t)j * d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += doi[c] * vj[c];
            dp[j] = acc;
            rowdot += p[j] * acc;
        }
        double *dqi = dq + (size_t)(rows ? r : i) * d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        for (int j = 0; j < Nk; ++j) {
            if (p[j] == 0.0) continue;
            double ds = p[j] * (dp[j] - rowdot);
            const double *kj = k + (size_t)j * d;
            for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
            if (dk && dv) {
                double *dkj = dk + (size_t)j * d, *dvj = dv + (size_t)j * d;
                for (int c = 0; c < d; ++c) {
                    dkj[c] += scale * ds * qi[c];
                    dvj[c] += p[j] * doi[c];
                }
            }
        }
    }
}

/* Full backward; parallel over heads (each head's dK/dV has one writer). */
int oracle_bwd(const double *q, const double *k, const double *v,
               const double *bias, const double *dO,
               double *dq, double *dk, double *dv,
               int B, int H, int Nq, int Nk, int d, double scale, int causal)
{
    const long BH = (long)B * H;
    int failed = 0;
    memset(dk, 0, sizeof(double) * (size_t)BH * Nk * d);
    memset(dv, 0, sizeof(double) * (size_t)BH * Nk * d);
#pragma omp parallel
    {
        size_t n = (size_t)(Nk > 0 ? Nk : 1);
        double *p = (double *)malloc(sizeof(double) * n);
        double *dp = (double *)malloc(sizeof(double) * n);
        if (!p || !dp) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            if (!p || !dp) continue;
            int b = (int)(bh / H);
            size_t qoff = (size_t)bh * Nq * d, koff = (size_t)bh * Nk * d;
            bwd_head(q + qoff, k + koff, v + koff,
                     bias ? bias + (size_t)b * Nk : NULL, dO + qoff,
                     dq + qoff, dk + koff, dv + koff, NULL, Nq,
                     Nq, Nk, d, scale, causal, p, dp);
        }
        free(p);
        free(dp);
    }
    return failed ? -1 : 0;
}

/* dQ for selected (head, row) pairs only: dq [n][d]. */
int oracle_bwd_dq_rows(const double *q, const double *k, const double *v,
                       const double *bias, const double *dO,
                       const long *heads, const int *rows, long n, double *dq,
                       int B, int H, int Nq, int Nk, int d, double scale, int causal)
{
    (void)B;
    int failed = 0;
#pragma omp parallel
    {
        size_t m = (size_t)(Nk > 0 ? Nk : 1);
        double *p = (double *)malloc(sizeof(double) * m);
        double *dp = (double *)malloc(sizeof(double) * m);
        if (!p || !dp) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < n; ++t) {
            if (!p || !dp) continue;
            long bh = heads[t];
            int b = (int)(bh / H);
            size_t qoff = (size_t)bh * Nq * d, koff = (size_t)bh * Nk * d;
            bwd_head(q + qoff, k + koff, v + koff,
                     bias ? bias + (size_t)b * Nk : NULL, dO + qoff,
                     dq + (size_t)t * d, NULL, NULL, rows + t, 1,
                     Nq, Nk, d, scale, causal, p, dp);
        }
        free(p);
        free(dp);
    }
    return failed ? -1 : 0;
}

/*
 * Backward contributions of selected query rows of ONE head, on the calling
 * thread: dq [nrows][d] (complete rows of dQ), and the part of dK, dV
 * ([Nk][d], accumulated into, caller zeroes them) that those rows produce.
 * Summed over all rows this is oracle_bwd; used to time the oracle on a
 * bounded sample of a workload.
 */
void oracle_bwd_head_rows(const double *q, const double *k, const double *v,
                          const double *bias, const double *dO, const int *rows, int nrows,
                          double *dq, double *dk, double *dv,
                          int Nq, int Nk, int d, double scale, int causal,
                          double *scratch /* 2 * Nk doubles */)
{
    bwd_head(q, k, v, bias, dO, dq, dk, dv, rows, nrows, Nq, Nk, d, scale, causal,
             scratch, scratch + Nk);
}

/* Forward of selected query rows of ONE head, on the calling thread:
 * o [nrows][d], lse [nrows]; scratch holds Nk doubles. */
void oracle_fwd_head_rows(const double *q, const double *k, const double *v,
                          const double *bias, const int *rows, int nrows,
                          double *o, double *lse, int Nq, int Nk, int d, double scale,
                          int causal, double *scratch)
{
    fwd_head_rows(q, k, v, bias, rows, 0, nrows, o, lse, Nq, Nk, d, scale, causal, scratch);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
