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
 * Parity pins for this file (closed forms, invariants, reductions to linear
 * attention, planted-mistake checks) live in tests/test_oracle_pins.py.
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
