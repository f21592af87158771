/*
 * gdn_oracle.c -- fp64 token-by-token oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference arm of bench.py may load this code.  It shares no
 * code with the CUDA path and is deliberately plain: one thread, fp64, no
 * blocking, no chunking, no reordering.
 *
 * What it computes ("Gated DeltaNet GPU并行实现", sections 2.1 and 2.2, and
 * the naive per-token loop of section 1.3 used there as the correctness
 * reference): per (sequence, head) a state S of shape d_v x d_k (row-major,
 * S[i*d_k + j], i over d_v, j over d_k) evolves over tokens t = 0..T-1 as
 *
 *     alpha_t = exp(log_alpha_t)
 *     S_t     = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t     = S_t q_t                    (the state AFTER token t's write)
 *
 * with S_{-1} = h0 (or zero) and hT = S_{T-1}.  Section 2.1 writes the delta
 * rule as S_{t-1} - beta (S_{t-1} k - v) k^T and expands it; the expansion is
 * the right-multiplication form above.  The gate of section 2.2 is a scalar
 * that scales the old state only (it multiplies the whole old-state term and
 * not the write beta v k^T).  The page also prints the erase factor on the
 * left, (I - beta k k^T) S; with S of shape d_v x d_k and o = S q only the
 * right-multiplication form type-checks when d_k != d_v, and it is what the
 * page's own expansion gives, so that is the form used here.  No 1/sqrt(d)
 * scaling is applied to q; the output is inclusive (o_t sees token t).
 *
 * The second half of the file is gated linear attention, the same
 * recurrence without the delta rule's erase term ("线性注意力机制与Gated
 * DeltaNet的优化实践", sections 2.2-2.3: the linear-attention state
 * S_i = S_{i-1} + k_i v_i^T and its gated form with a forget gate and an
 * update gate, both scalars here):
 *
 *     S_t = alpha_t * S_{t-1} + beta_t v_t k_t^T,     o_t = S_t q_t
 *
 * (alpha = beta = 1 is plain linear attention), in the same layouts.
 *
 * The third part takes a gate per key dimension ("Gated DeltaNet GPU并行实现",
 * section 2.2: with a per-dimension or diagonal gate the affine map's
 * coefficient matrix gains a diagonal factor).  Reading: the diagonal factor
 * acts on the old state first, as the scalar gate does,
 *
 *     S_t = (S_{t-1} diag(alpha_t)) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *
 * alpha_t = exp(log_alpha_t) with log_alpha_t a d_k-vector; with the erase
 * term off it is gated linear attention with a vector gate.
 *
 * The last part is the gradient of the first two loops.  No page writes the
 * backward pass of the delta rule out; "企业官网建设流程全解析" (a page on
 * linear-attention training) recomputes the recurrent state in the backward
 * pass instead of storing it (sections 2 and 4.3) and checks gradients
 * numerically (section 5.3).  The gradient here is the plain definition: for
 * output weights dO [T][dv] and dhT [dv][dk] it returns the gradient of
 *
 *     L = sum_t dO_t . o_t + <dhT, hT>
 *
 * with respect to q, k, v, log_alpha, beta and h0, by reverse-mode
 * differentiation of the token loop: the forward states S_{-1..T-1} are kept,
 * then the tokens are walked backwards with the adjoint dS of the current
 * state.
 *
 * Parity pins for this file (closed forms, invariants, reductions to linear
 * attention, finite differences, planted-mistake checks) live in
 * tests/test_oracle_pins.py; examples worked by hand are in tests/golden/,
 * checked by tests/test_golden.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/*
 * One (sequence, head).  q,k: [T][dk]; v: [T][dv]; la, beta: [T];
 * h0, hT: [dv][dk] (h0 may be NULL = zero state, hT may be NULL = not
 * written); o: [T][dv] (may be NULL).  S and kS are caller scratch of dv*dk
 * and dv doubles.
 */
static void oracle_one(const double *q, const double *k, const double *v,
                       const double *la, const double *beta,
                       const double *h0, double *o, double *hT,
                       long T, long dk, long dv, double *S, double *kS)
{
    long t, i, j;
    if (h0)
        memcpy(S, h0, sizeof(double) * (size_t)(dv * dk));
    else
        memset(S, 0, sizeof(double) * (size_t)(dv * dk));

    for (t = 0; t < T; ++t) {
        const double *kt = k + t * dk;
        const double *vt = v + t * dv;
        const double *qt = q + t * dk;
        const double a = exp(la[t]);
        const double b = beta[t];

        /* kS = S_{t-1} k_t  (a d_v vector) */
        for (i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (j = 0; j < dk; ++j)
                acc += S[i * dk + j] * kt[j];
            kS[i] = acc;
        }
        /* S_t = a*(S_{t-1} - b*(S_{t-1} k_t) k_t^T) + b*v_t k_t^T */
        for (i = 0; i < dv; ++i) {
            for (j = 0; j < dk; ++j) {
                double s = S[i * dk + j];
                S[i * dk + j] = a * (s - b * kS[i] * kt[j]) + b * vt[i] * kt[j];
            }
        }
        /* o_t = S_t q_t */
        if (o) {
            for (i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (j = 0; j < dk; ++j)
                    acc += S[i * dk + j] * qt[j];
                o[t * dv + i] = acc;
            }
        }
    }
    if (hT)
        memcpy(hT, S, sizeof(double) * (size_t)(dv * dk));
}

/*
 * Dense batch: q,k [B][H][T][dk]; v, o [B][H][T][dv]; log_alpha, beta
 * [B][H][T]; h0, hT [B][H][dv][dk].  Returns 0, or -1 on a bad argument or
 * allocation failure.
 */
int gdn_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta,
                   const double *h0, double *o, double *hT,
                   long B, long H, long T, long dk, long dv)
{
    long bh;
    double *S, *kS;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    kS = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !kS) {
        free(S);
        free(kS);
        return -1;
    }
    for (bh = 0; bh < B * H; ++bh) {
        oracle_one(q + bh * T * dk, k + bh * T * dk, v + bh * T * dv,
                   log_alpha + bh * T, beta + bh * T,
                   h0 ? h0 + bh * dv * dk : NULL,
                   o ? o + bh * T * dv : NULL,
                   hT ? hT + bh * dv * dk : NULL,
                   T, dk, dv, S, kS);
    }
    free(S);
    free(kS);
    return 0;
}

/*
 * Packed variable-length batch: N sequences concatenated along one token
 * axis of length T_total, sequence n occupying tokens
 * [cu_seqlens[n], cu_seqlens[n+1]).  q,k [H][T_total][dk]; v, o
 * [H][T_total][dv]; log_alpha, beta [H][T_total]; h0, hT [N][H][dv][dk].
 * Sequences never interact; each starts from its own h0.
 */
int gdn_oracle_fwd_varlen(const double *q, const double *k, const double *v,
                          const double *log_alpha, const double *beta,
                          const double *h0, double *o, double *hT,
                          const long *cu_seqlens, long N, long H, long T_total,
                          long dk, long dv)
{
    long n, h;
    double *S, *kS;
    if (N < 0 || H < 0 || T_total < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total))
        return -1;
    for (n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    kS = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !kS) {
        free(S);
        free(kS);
        return -1;
    }
    for (n = 0; n < N; ++n) {
        long t0 = cu_seqlens[n];
        long len = cu_seqlens[n + 1] - t0;
        for (h = 0; h < H; ++h) {
            long row = h * T_total + t0;
            oracle_one(q + row * dk, k + row * dk, v + row * dv,
                       log_alpha + row, beta + row,
                       h0 ? h0 + (n * H + h) * dv * dk : NULL,
                       o ? o + row * dv : NULL,
                       hT ? hT + (n * H + h) * dv * dk : NULL,
                       len, dk, dv, S, kS);
        }
    }
    free(S);
    free(kS);
    return 0;
}

/*
 * Gated linear attention, one (sequence, head): the loop above with the
 * erase term left out.  Same arguments; S is caller scratch of dv*dk doubles.
 */
static void oracle_one_gla(const double *q, const double *k, const double *v,
                           const double *la, const double *beta,
                           const double *h0, double *o, double *hT,
                           long T, long dk, long dv, double *S)
{
    long t, i, j;
    if (h0)
        memcpy(S, h0, sizeof(double) * (size_t)(dv * dk));
    else
        memset(S, 0, sizeof(double) * (size_t)(dv * dk));
    for (t = 0; t < T; ++t) {
        const double *kt = k + t * dk;
        const double *vt = v + t * dv;
        const double *qt = q + t * dk;
        const double g = exp(la[t]);
        const double w = beta[t];
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                S[i * dk + j] = g * S[i * dk + j] + w * vt[i] * kt[j];
        if (o) {
            for (i = 0; i < dv; ++i) {
                double sum = 0.0;
                for (j = 0; j < dk; ++j)
                    sum += S[i * dk + j] * qt[j];
                o[t * dv + i] = sum;
            }
        }
    }
    if (hT)
        memcpy(hT, S, sizeof(double) * (size_t)(dv * dk));
}

/* Dense batch, gated linear attention (layouts as gdn_oracle_fwd). */
int gdn_oracle_gla_fwd(const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *beta,
                       const double *h0, double *o, double *hT,
                       long B, long H, long T, long dk, long dv)
{
    long bh;
    double *S;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    if (!S)
        return -1;
    for (bh = 0; bh < B * H; ++bh)
        oracle_one_gla(q + bh * T * dk, k + bh * T * dk, v + bh * T * dv,
                       log_alpha + bh * T, beta + bh * T,
                       h0 ? h0 + bh * dv * dk : NULL,
                       o ? o + bh * T * dv : NULL,
                       hT ? hT + bh * dv * dk : NULL,
                       T, dk, dv, S);
    free(S);
    return 0;
}

/* Packed batch, gated linear attention (layouts as gdn_oracle_fwd_varlen). */
int gdn_oracle_gla_fwd_varlen(const double *q, const double *k, const double *v,
                              const double *log_alpha, const double *beta,
                              const double *h0, double *o, double *hT,
                              const long *cu_seqlens, long N, long H, long T_total,
                              long dk, long dv)
{
    long n, h;
    double *S;
    if (N < 0 || H < 0 || T_total < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total))
        return -1;
    for (n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    if (!S)
        return -1;
    for (n = 0; n < N; ++n) {
        long s0 = cu_seqlens[n];
        long len = cu_seqlens[n + 1] - s0;
        for (h = 0; h < H; ++h) {
            long rw = h * T_total + s0;
            oracle_one_gla(q + rw * dk, k + rw * dk, v + rw * dv,
                           log_alpha + rw, beta + rw,
                           h0 ? h0 + (n * H + h) * dv * dk : NULL,
                           o ? o + rw * dv : NULL,
                           hT ? hT + (n * H + h) * dv * dk : NULL,
                           len, dk, dv, S);
        }
    }
    free(S);
    return 0;
}

/*
 * Per-dimension gate, one (sequence, head).  la: [T][dk]; erase = 0 leaves
 * the erase term out.  Otherwise as oracle_one.
 */
static void oracle_one_vg(const double *q, const double *k, const double *v,
                          const double *la, const double *beta,
                          const double *h0, double *o, double *hT,
                          long T, long dk, long dv, long erase, double *S, double *Sk)
{
    long t, i, j;
    if (h0)
        memcpy(S, h0, sizeof(double) * (size_t)(dv * dk));
    else
        memset(S, 0, sizeof(double) * (size_t)(dv * dk));
    for (t = 0; t < T; ++t) {
        const double *kt = k + t * dk;
        const double *vt = v + t * dv;
        const double *qt = q + t * dk;
        const double *lat = la + t * dk;
        const double bt = beta[t];
        /* S <- S diag(alpha_t): column j scaled by exp(la_t[j]) */
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                S[i * dk + j] *= exp(lat[j]);
        /* S <- S (I - b k k^T) + b v k^T */
        for (i = 0; i < dv; ++i) {
            double dot = 0.0;
            for (j = 0; j < dk; ++j)
                dot += S[i * dk + j] * kt[j];
            Sk[i] = erase ? dot : 0.0;
        }
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                S[i * dk + j] += bt * (vt[i] - Sk[i]) * kt[j];
        if (o) {
            for (i = 0; i < dv; ++i) {
                double out = 0.0;
                for (j = 0; j < dk; ++j)
                    out += S[i * dk + j] * qt[j];
                o[t * dv + i] = out;
            }
        }
    }
    if (hT)
        memcpy(hT, S, sizeof(double) * (size_t)(dv * dk));
}

/* Dense batch, per-dimension gate: log_alpha [B][H][T][dk], rest as gdn_oracle_fwd. */
int gdn_oracle_vg_fwd(const double *q, const double *k, const double *v,
                      const double *log_alpha, const double *beta,
                      const double *h0, double *o, double *hT,
                      long B, long H, long T, long dk, long dv, long erase)
{
    long bh;
    double *S, *Sk;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    Sk = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !Sk) {
        free(S);
        free(Sk);
        return -1;
    }
    for (bh = 0; bh < B * H; ++bh)
        oracle_one_vg(q + bh * T * dk, k + bh * T * dk, v + bh * T * dv,
                      log_alpha + bh * T * dk, beta + bh * T,
                      h0 ? h0 + bh * dv * dk : NULL,
                      o ? o + bh * T * dv : NULL,
                      hT ? hT + bh * dv * dk : NULL,
                      T, dk, dv, erase, S, Sk);
    free(S);
    free(Sk);
    return 0;
}

/* Packed batch, per-dimension gate: log_alpha [H][T_total][dk]. */
int gdn_oracle_vg_fwd_varlen(const double *q, const double *k, const double *v,
                             const double *log_alpha, const double *beta,
                             const double *h0, double *o, double *hT,
                             const long *cu_seqlens, long N, long H, long T_total,
                             long dk, long dv, long erase)
{
    long n, h;
    double *S, *Sk;
    if (N < 0 || H < 0 || T_total < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total))
        return -1;
    for (n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -1;
    S = (double *)malloc(sizeof(double) * (size_t)(dv * dk));
    Sk = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !Sk) {
        free(S);
        free(Sk);
        return -1;
    }
    for (n = 0; n < N; ++n) {
        long first = cu_seqlens[n];
        long len = cu_seqlens[n + 1] - first;
        for (h = 0; h < H; ++h) {
            long at = h * T_total + first;
            oracle_one_vg(q + at * dk, k + at * dk, v + at * dv,
                          log_alpha + at * dk, beta + at,
                          h0 ? h0 + (n * H + h) * dv * dk : NULL,
                          o ? o + at * dv : NULL,
                          hT ? hT + (n * H + h) * dv * dk : NULL,
                          len, dk, dv, erase, S, Sk);
        }
    }
    free(S);
    free(Sk);
    return 0;
}

/*
 * Gradient of one (sequence, head); erase = 0 differentiates the gated
 * linear attention loop instead.  Layouts as oracle_one; dout [T][dv];
 * dhT, h0 and dh0 may be NULL (zero weight / zero state / not written).
 * Per token t, with X = S_{t-1}, a = alpha_t, b = beta_t and dS the adjoint
 * of S_t (which already holds dO_t q_t^T from o_t = S_t q_t):
 *     dq_t       = S_t^T dO_t
 *     dv_t       = b dS k_t
 *     dbeta_t    = (dS k_t) . (v_t - a X k_t)            [erase]
 *                  (dS k_t) . v_t                        [no erase]
 *     dalpha_t   = <dS, X> - b (dS k_t) . (X k_t)        [no erase: <dS, X>]
 *     dk_t       = b dS^T v_t - a b (X^T dS k_t + dS^T X k_t)   [no erase: b dS^T v_t]
 *     dS_{t-1}   = a dS (I - b k_t k_t^T)                [no erase: a dS]
 *     dlog_alpha_t = a dalpha_t
 * Returns 0, or -1 when the state history cannot be allocated.
 */
static int oracle_one_bwd(const double *q, const double *k, const double *v,
                          const double *la, const double *beta, const double *h0,
                          const double *dout, const double *dhT,
                          double *dq, double *dk_, double *dv_, double *dla,
                          double *dbeta, double *dh0,
                          long T, long dk, long dv, long erase)
{
    const long n = dv * dk;
    long t, i, j;
    double *St = (double *)malloc(sizeof(double) * (size_t)((T + 1) * n));
    double *dS = (double *)malloc(sizeof(double) * (size_t)n);
    double *Xk = (double *)malloc(sizeof(double) * (size_t)dv);
    double *dSk = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!St || !dS || !Xk || !dSk) {
        free(St);
        free(dS);
        free(Xk);
        free(dSk);
        return -1;
    }
    /* forward, keeping every state: St + (t+1)*n holds S_t, St holds S_{-1} */
    if (h0)
        memcpy(St, h0, sizeof(double) * (size_t)n);
    else
        memset(St, 0, sizeof(double) * (size_t)n);
    for (t = 0; t < T; ++t) {
        const double *X = St + t * n;
        double *Y = St + (t + 1) * n;
        const double *kt = k + t * dk, *vt = v + t * dv;
        const double a = exp(la[t]), b = beta[t];
        for (i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (j = 0; j < dk; ++j)
                acc += X[i * dk + j] * kt[j];
            Xk[i] = erase ? acc : 0.0;
        }
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                Y[i * dk + j] = a * (X[i * dk + j] - b * Xk[i] * kt[j]) + b * vt[i] * kt[j];
    }
    /* backward */
    if (dhT)
        memcpy(dS, dhT, sizeof(double) * (size_t)n);
    else
        memset(dS, 0, sizeof(double) * (size_t)n);
    for (t = T - 1; t >= 0; --t) {
        const double *X = St + t * n;
        const double *Y = St + (t + 1) * n;
        const double *kt = k + t * dk, *vt = v + t * dv, *qt = q + t * dk;
        const double *dot = dout + t * dv;
        const double a = exp(la[t]), b = beta[t];
        double sx = 0.0, db = 0.0, cross = 0.0;
        /* o_t = S_t q_t */
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                dS[i * dk + j] += dot[i] * qt[j];
        for (j = 0; j < dk; ++j) {
            double acc = 0.0;
            for (i = 0; i < dv; ++i)
                acc += Y[i * dk + j] * dot[i];
            dq[t * dk + j] = acc;
        }
        for (i = 0; i < dv; ++i) {
            double a1 = 0.0, a2 = 0.0;
            for (j = 0; j < dk; ++j) {
                a1 += dS[i * dk + j] * kt[j];
                a2 += X[i * dk + j] * kt[j];
                sx += dS[i * dk + j] * X[i * dk + j];
            }
            dSk[i] = a1;
            Xk[i] = a2;
        }
        for (i = 0; i < dv; ++i) {
            dv_[t * dv + i] = b * dSk[i];
            db += dSk[i] * (erase ? vt[i] - a * Xk[i] : vt[i]);
            cross += dSk[i] * Xk[i];
        }
        dbeta[t] = db;
        dla[t] = a * (erase ? sx - b * cross : sx);
        for (j = 0; j < dk; ++j) {
            double acc = 0.0;
            for (i = 0; i < dv; ++i) {
                acc += b * dS[i * dk + j] * vt[i];
                if (erase)
                    acc -= a * b * (X[i * dk + j] * dSk[i] + dS[i * dk + j] * Xk[i]);
            }
            dk_[t * dk + j] = acc;
        }
        for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j)
                dS[i * dk + j] = a * (dS[i * dk + j] - (erase ? b * dSk[i] * kt[j] : 0.0));
    }
    if (dh0)
        memcpy(dh0, dS, sizeof(double) * (size_t)n);
    free(St);
    free(dS);
    free(Xk);
    free(dSk);
    return 0;
}

/*
 * Dense batch gradient: inputs as gdn_oracle_fwd, dout [B][H][T][dv], dhT
 * [B][H][dv][dk] (or NULL); gradients in the layouts of their inputs.
 */
int gdn_oracle_bwd(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta, const double *h0,
                   const double *dout, const double *dhT,
                   double *dq, double *dk_, double *dv_, double *dla, double *dbeta,
                   double *dh0, long B, long H, long T, long dk, long dv, long erase)
{
    long bh;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
        return -1;
    for (bh = 0; bh < B * H; ++bh)
        if (oracle_one_bwd(q + bh * T * dk, k + bh * T * dk, v + bh * T * dv,
                           log_alpha + bh * T, beta + bh * T,
                           h0 ? h0 + bh * dv * dk : NULL, dout + bh * T * dv,
                           dhT ? dhT + bh * dv * dk : NULL,
                           dq + bh * T * dk, dk_ + bh * T * dk, dv_ + bh * T * dv,
                           dla + bh * T, dbeta + bh * T,
                           dh0 ? dh0 + bh * dv * dk : NULL, T, dk, dv, erase))
            return -1;
    return 0;
}

/* Packed batch gradient: layouts as gdn_oracle_fwd_varlen. */
int gdn_oracle_bwd_varlen(const double *q, const double *k, const double *v,
                          const double *log_alpha, const double *beta, const double *h0,
                          const double *dout, const double *dhT,
                          double *dq, double *dk_, double *dv_, double *dla, double *dbeta,
                          double *dh0, const long *cu_seqlens, long N, long H, long T_total,
                          long dk, long dv, long erase)
{
    long n, h;
    if (N < 0 || H < 0 || T_total < 0 || dk <= 0 || dv <= 0)
        return -1;
    if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total))
        return -1;
    for (n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -1;
    for (n = 0; n < N; ++n) {
        long s0 = cu_seqlens[n];
        long len = cu_seqlens[n + 1] - s0;
        for (h = 0; h < H; ++h) {
            long rw = h * T_total + s0;
            long st = (n * H + h) * dv * dk;
            if (oracle_one_bwd(q + rw * dk, k + rw * dk, v + rw * dv, log_alpha + rw,
                               beta + rw, h0 ? h0 + st : NULL, dout + rw * dv,
                               dhT ? dhT + st : NULL, dq + rw * dk, dk_ + rw * dk,
                               dv_ + rw * dv, dla + rw, dbeta + rw, dh0 ? dh0 + st : NULL,
                               len, dk, dv, erase))
                return -1;
        }
    }
    return 0;
}
