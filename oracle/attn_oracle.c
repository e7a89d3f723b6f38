/*
 * FP64 CPU oracle for exact softmax attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this code.  It shares
 * no code, header, table or helper with the CUDA path and never calls it.
 *
 * What it computes (one head; Q, K, V, dO are [N, d] row-major, upcast to
 * double from the rounded 16-bit inputs by the caller):
 *
 *   Forward ("Writing Speed-of-Light Attention Backward Kernel for 5090 in
 *   CUDA", section "Mathematical Formulation", forward equations):
 *     S   = scale * Q K^T + M        M_ij = -inf if (causal and j > i) else 0
 *     L_i = log sum_j exp(S_ij)      (natural log; evaluated as
 *                                     m_i + log sum_j exp(S_ij - m_i) with
 *                                     m_i = max_j S_ij, the same number)
 *     P   = exp(S - L)
 *     O   = P V
 *
 *   Backward (same page, same section, "The complete backward pass"):
 *     D   = rowsum(dO o O)
 *     dV  = P^T dO
 *     dP  = dO V^T
 *     dS  = P o (dP - D 1^T)
 *     dQ  = scale * dS K
 *     dK  = scale * dS^T Q
 *   The page writes 1/sqrt(d) in dQ and dK; the caller's `scale` replaces it
 *   (it is 1/sqrt(d) on every workload).  D uses the oracle's own O.
 *
 * The work is done one query row i at a time: row i of S, L_i, row i of P,
 * O_i, D_i, row i of dP and dS, dQ_i; the sums over i that make dV_j and
 * dK_j are accumulated in increasing i.  That is the plain evaluation order
 * of the equations above, with no blocking or reordering.
 *
 * Every entry point returns 0 on success and a negative number on bad sizes
 * or an allocation failure.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Mask term M_ij of the forward equation. */
static double mask_term(int causal, long i, long j)
{
    return (causal && j > i) ? -INFINITY : 0.0;
}

/* Row i of S into s[0..N), returns max_j S_ij. */
static double score_row(const double *q, const double *k, long N, long d,
                        double scale, int causal, long i, double *s)
{
    double m = -INFINITY;
    for (long j = 0; j < N; ++j) {
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += q[i * d + c] * k[j * d + c];
        s[j] = scale * dot + mask_term(causal, i, j);
        if (s[j] > m) m = s[j];
    }
    return m;
}

/* L_i from row i of S (natural log-sum-exp, max-shifted for range). */
static double logsumexp_row(const double *s, long N, double m)
{
    double acc = 0.0;
    for (long j = 0; j < N; ++j) acc += exp(s[j] - m);
    return m + log(acc);
}

/* Row i of the forward: P_i (into p), O_i, L_i. */
static void forward_row(const double *q, const double *k, const double *v,
                        long N, long d, double scale, int causal, long i,
                        double *s, double *p, double *o_i, double *lse_i)
{
    double m = score_row(q, k, N, d, scale, causal, i, s);
    double L = logsumexp_row(s, N, m);
    *lse_i = L;
    for (long j = 0; j < N; ++j) p[j] = exp(s[j] - L);
    for (long c = 0; c < d; ++c) o_i[c] = 0.0;
    for (long j = 0; j < N; ++j) {
        if (p[j] == 0.0) continue; /* exact zero adds nothing */
        for (long c = 0; c < d; ++c) o_i[c] += p[j] * v[j * d + c];
    }
}

/* Row i of the backward: dP_i, D_i, dS_i (into ds), dQ_i. */
static void backward_row(const double *q, const double *k, const double *v,
                         const double *dout, long N, long d, double scale,
                         long i, const double *p, const double *o_i,
                         double *ds, double *dq_i, double *D_i)
{
    (void)q;
    double D = 0.0;
    for (long c = 0; c < d; ++c) D += dout[i * d + c] * o_i[c];
    *D_i = D;
    for (long j = 0; j < N; ++j) {
        double dp = 0.0;
        for (long c = 0; c < d; ++c) dp += dout[i * d + c] * v[j * d + c];
        ds[j] = p[j] * (dp - D);
    }
    for (long c = 0; c < d; ++c) dq_i[c] = 0.0;
    for (long j = 0; j < N; ++j) {
        if (ds[j] == 0.0) continue;
        for (long c = 0; c < d; ++c) dq_i[c] += ds[j] * k[j * d + c];
    }
    for (long c = 0; c < d; ++c) dq_i[c] *= scale;
}

static int bad_sizes(long BH, long N, long d)
{
    return BH < 0 || N < 0 || d <= 0;
}

/*
 * Forward over BH independent heads.  q, k, v, o: [BH, N, d]; lse: [BH, N].
 */
int oracle_attn_fwd(long BH, long N, long d, double scale, int causal,
                    const double *q, const double *k, const double *v,
                    double *o, double *lse)
{
    if (bad_sizes(BH, N, d)) return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long h = 0; h < BH; ++h) {
        double *s = malloc(sizeof(double) * (size_t)(N ? N : 1));
        double *p = malloc(sizeof(double) * (size_t)(N ? N : 1));
        if (!s || !p) { err |= 1; free(s); free(p); continue; }
        const double *qh = q + h * N * d, *kh = k + h * N * d, *vh = v + h * N * d;
        for (long i = 0; i < N; ++i)
            forward_row(qh, kh, vh, N, d, scale, causal, i, s, p,
                        o + (h * N + i) * d, lse + h * N + i);
        free(s);
        free(p);
    }
    return err ? -2 : 0;
}

/*
 * Forward and backward over BH independent heads.  Inputs q, k, v, dout:
 * [BH, N, d].  Outputs dq, dk, dv: [BH, N, d].  Optional outputs (may be
 * NULL): o [BH, N, d], lse [BH, N], delta [BH, N] (the D vector).
 */
int oracle_attn_bwd(long BH, long N, long d, double scale, int causal,
                    const double *q, const double *k, const double *v,
                    const double *dout, double *dq, double *dk, double *dv,
                    double *o, double *lse, double *delta)
{
    if (bad_sizes(BH, N, d)) return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long h = 0; h < BH; ++h) {
        size_t n1 = (size_t)(N ? N : 1);
        double *s = malloc(sizeof(double) * n1);
        double *p = malloc(sizeof(double) * n1);
        double *ds = malloc(sizeof(double) * n1);
        double *o_i = malloc(sizeof(double) * (size_t)d);
        if (!s || !p || !ds || !o_i) {
            err |= 1; free(s); free(p); free(ds); free(o_i); continue;
        }
        const double *qh = q + h * N * d, *kh = k + h * N * d;
        const double *vh = v + h * N * d, *doh = dout + h * N * d;
        double *dqh = dq + h * N * d, *dkh = dk + h * N * d, *dvh = dv + h * N * d;
        memset(dkh, 0, sizeof(double) * (size_t)(N * d));
        memset(dvh, 0, sizeof(double) * (size_t)(N * d));
        for (long i = 0; i < N; ++i) {
            double L, D;
            forward_row(qh, kh, vh, N, d, scale, causal, i, s, p, o_i, &L);
            backward_row(qh, kh, vh, doh, N, d, scale, i, p, o_i, ds,
                         dqh + i * d, &D);
            /* dV_j += P_ij dO_i ;  dK_j += scale * dS_ij Q_i */
            for (long j = 0; j < N; ++j) {
                if (p[j] != 0.0)
                    for (long c = 0; c < d; ++c) dvh[j * d + c] += p[j] * doh[i * d + c];
                if (ds[j] != 0.0)
                    for (long c = 0; c < d; ++c) dkh[j * d + c] += scale * ds[j] * qh[i * d + c];
            }
            if (o) memcpy(o + (h * N + i) * d, o_i, sizeof(double) * (size_t)d);
            if (lse) lse[h * N + i] = L;
            if (delta) delta[h * N + i] = D;
        }
        free(s); free(p); free(ds); free(o_i);
    }
    return err ? -2 : 0;
}

/*
 * Selected query rows of one head: O_i, L_i and dQ_i for i in rows[0..nrows).
 * Each needs only row i of S, P, dP and dS, so this is O(N d) per row and
 * serves as the sampled-output oracle at sizes where a whole head is too
 * slow.  q, k, v, dout: [N, d].  o_rows, dq_rows: [nrows, d]; lse_rows:
 * [nrows].  dout and dq_rows may both be NULL to skip the backward part.
 */
int oracle_attn_rows(long N, long d, double scale, int causal,
                     const double *q, const double *k, const double *v,
                     const double *dout, long nrows, const long *rows,
                     double *o_rows, double *lse_rows, double *dq_rows)
{
    if (bad_sizes(1, N, d) || nrows < 0) return -1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long r = 0; r < nrows; ++r) {
        size_t n1 = (size_t)(N ? N : 1);
        double *s = malloc(sizeof(double) * n1);
        double *p = malloc(sizeof(double) * n1);
        double *ds = malloc(sizeof(double) * n1);
        if (!s || !p || !ds) { err |= 1; free(s); free(p); free(ds); continue; }
        long i = rows[r];
        forward_row(q, k, v, N, d, scale, causal, i, s, p, o_rows + r * d, lse_rows + r);
        if (dout && dq_rows) {
            double D;
            backward_row(q, k, v, dout, N, d, scale, i, p, o_rows + r * d, ds,
                         dq_rows + r * d, &D);
        }
        free(s); free(p); free(ds);
    }
    return err ? -2 : 0;
}

/*
 * Forward and backward restricted to the listed query rows of ONE head: the
 * same per-row work as oracle_attn_bwd, for rows[0..nrows) only.  dq_rows
 * [nrows, d] gets dQ_i; dk_part and dv_part [N, d] get the contributions of
 * just these rows to dK and dV (the sums over i of oracle_attn_bwd, restricted
 * to the listed i).  Used to time a bounded, representative sample of a large
 * workload; not parallel (callers run one head per thread).
 */
int oracle_attn_bwd_rowset(long N, long d, double scale, int causal,
                           const double *q, const double *k, const double *v,
                           const double *dout, long nrows, const long *rows,
                           double *dq_rows, double *dk_part, double *dv_part)
{
    if (bad_sizes(1, N, d) || nrows < 0) return -1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    size_t n1 = (size_t)(N ? N : 1);
    double *s = malloc(sizeof(double) * n1);
    double *p = malloc(sizeof(double) * n1);
    double *ds = malloc(sizeof(double) * n1);
    double *o_i = malloc(sizeof(double) * (size_t)d);
    if (!s || !p || !ds || !o_i) { free(s); free(p); free(ds); free(o_i); return -2; }
    memset(dk_part, 0, sizeof(double) * (size_t)(N * d));
    memset(dv_part, 0, sizeof(double) * (size_t)(N * d));
    for (long r = 0; r < nrows; ++r) {
        long i = rows[r];
        double L, D;
        forward_row(q, k, v, N, d, scale, causal, i, s, p, o_i, &L);
        backward_row(q, k, v, dout, N, d, scale, i, p, o_i, ds, dq_rows + r * d, &D);
        for (long j = 0; j < N; ++j) {
            if (p[j] != 0.0)
                for (long c = 0; c < d; ++c) dv_part[j * d + c] += p[j] * dout[i * d + c];
            if (ds[j] != 0.0)
                for (long c = 0; c < d; ++c) dk_part[j * d + c] += scale * ds[j] * q[i * d + c];
        }
    }
    free(s); free(p); free(ds); free(o_i);
    return 0;
}

/*
 * Whole P and dS matrices of one head ([N, N] each), for invariant checks on
 * tiny inputs.  dout may be NULL, in which case ds is not written.
 */
int oracle_attn_probs(long N, long d, double scale, int causal,
                      const double *q, const double *k, const double *v,
                      const double *dout, double *P, double *dS)
{
    if (bad_sizes(1, N, d)) return -1;
    size_t n1 = (size_t)(N ? N : 1);
    double *s = malloc(sizeof(double) * n1);
    double *o_i = malloc(sizeof(double) * (size_t)d);
    double *dq_i = malloc(sizeof(double) * (size_t)d);
    if (!s || !o_i || !dq_i) { free(s); free(o_i); free(dq_i); return -2; }
    for (long i = 0; i < N; ++i) {
        double L, D;
        forward_row(q, k, v, N, d, scale, causal, i, s, P + i * N, o_i, &L);
        if (dout && dS)
            backward_row(q, k, v, dout, N, d, scale, i, P + i * N, o_i,
                         dS + i * N, dq_i, &D);
    }
    free(s); free(o_i); free(dq_i);
    return 0;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
