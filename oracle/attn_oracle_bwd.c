/*
 * CPU oracle for the attention backward.  TEST INFRASTRUCTURE ONLY (same rules
 * as attn_oracle.c: only the tests, the smoke check and the bench's CPU leg
 * use it; it shares nothing with the CUDA path).
 *
 * What it computes: the gradients of L = sum_{i,d} dO_id * O_id with respect
 * to Q, K and V, where O = softmax(scale * Q K^T [+ causal]) V is the forward
 * of "[GPU] Deep Learning for HPC" (bkkhyunn.github.io, section "Flash
 * Attention").  The pages call the backward an order of magnitude harder than
 * the forward and point at TMA's asynchronous reductions for it
 * ("GPUの爆発的な性能向上", ja.news.hada.io topic 14783, sections "アドレス生成と
 * TMA" and the closing discussion), but print no formula; the formula here is
 * the chain rule through the softmax, written out:
 *
 *   p_ij  = exp(s_ij - m_i) / l_i                  (two-pass softmax, as forward)
 *   o_i   = sum_j p_ij v_j
 *   dp_ij = sum_d dO_id v_jd                       (dL/dp_ij)
 *   D_i   = sum_j p_ij dp_ij                       (softmax Jacobian term)
 *   ds_ij = p_ij (dp_ij - D_i)                     (dL/ds_ij)
 *   dq_i  = scale sum_j ds_ij k_j
 *   dk_j  = scale sum_i ds_ij q_i
 *   dv_j  = sum_i p_ij dO_i
 *
 * Masking and lengths as the forward oracle: causal key j is visible to query
 * i iff j <= i + (Nk - Nq); a query with no visible key has o = 0, lse = -inf,
 * D = 0 and contributes nothing.  All arithmetic is double precision; every sum
 * runs in increasing index order (dk, dv accumulate over queries i in order).
 * (b, h) slices are independent and spread over OpenMP threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16_b(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One (b, h) slice.  q, dout [Nq*D]; k, v [Nk*D]; outputs dq [Nq*D], dk, dv
 * [Nk*D], delta, lse [Nq], o [Nq*D].  s, p, dp: scratch of Nk doubles. */
static void bwd_slice(const double *q, const double *k, const double *v, const double *dout,
                      double *dq, double *dk, double *dv, double *delta, double *o, double *lse,
                      int64_t Nq, int64_t Nk, int64_t D, int causal, double scale,
                      double *s, double *p, double *dp) {
    int64_t i, j, d;
    for (j = 0; j < Nk * D; ++j) {
        dk[j] = 0.0;
        dv[j] = 0.0;
    }
    for (i = 0; i < Nq; ++i) {
        const double *qi = q + i * D, *doi = dout + i * D;
        double *dqi = dq + i * D, *oi = o + i * D;
        int64_t n_vis = Nk;
        if (causal) {
            n_vis = i + (Nk - Nq) + 1;
            if (n_vis > Nk) n_vis = Nk;
            if (n_vis < 0) n_vis = 0;
        }
        for (d = 0; d < D; ++d) {
            dqi[d] = 0.0;
            oi[d] = 0.0;
        }
        if (n_vis == 0) {
            delta[i] = 0.0;
            lse[i] = -INFINITY;
            continue;
        }
        for (j = 0; j < n_vis; ++j) {
            double a = 0.0;
            for (d = 0; d < D; ++d) a += qi[d] * k[j * D + d];
            s[j] = scale * a;
        }
        double m = s[0];
        for (j = 1; j < n_vis; ++j)
            if (s[j] > m) m = s[j];
        double l = 0.0;
        for (j = 0; j < n_vis; ++j) l += exp(s[j] - m);
        for (j = 0; j < n_vis; ++j) p[j] = exp(s[j] - m) / l;
        lse[i] = m + log(l);
        for (j = 0; j < n_vis; ++j)
            for (d = 0; d < D; ++d) oi[d] += p[j] * v[j * D + d];
        double dl = 0.0;
        for (j = 0; j < n_vis; ++j) {
            double a = 0.0;
            for (d = 0; d < D; ++d) a += doi[d] * v[j * D + d];
            dp[j] = a;
            dl += p[j] * a;
        }
        delta[i] = dl;
        for (j = 0; j < n_vis; ++j) {
            const double ds = p[j] * (dp[j] - dl);
            for (d = 0; d < D; ++d) {
                dqi[d] += scale * ds * k[j * D + d];
                dk[j * D + d] += scale * ds * qi[d];
                dv[j * D + d] += p[j] * doi[d];
            }
        }
    }
}

static int nthreads_or_all(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Backward from double inputs.  q, dout, dq, o [B*H*Nq*D]; k, v, dk, dv
 * [B*H*Nk*D]; delta, lse [B*H*Nq].  Returns 0, or -1 on a bad argument or a
 * failed allocation. */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *dout,
                        double *dq, double *dk, double *dv, double *delta, double *o, double *lse,
                        int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal,
                        double scale, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !delta || !o || !lse) return -1;
    if (B < 0 || H < 0 || Nq < 1 || Nk < 1 || D < 1) return -1;
    const int64_t BH = B * H;
    int failed = 0;
    const int nt = nthreads_or_all(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt) reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *p = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Nk);
        if (!s || !p || !dp) {
            failed = 1;
        } else {
            int64_t bh;
#pragma omp for schedule(dynamic, 1)
            for (bh = 0; bh < BH; ++bh)
                bwd_slice(q + bh * Nq * D, k + bh * Nk * D, v + bh * Nk * D, dout + bh * Nq * D,
                          dq + bh * Nq * D, dk + bh * Nk * D, dv + bh * Nk * D, delta + bh * Nq,
                          o + bh * Nq * D, lse + bh * Nq, Nq, Nk, D, causal, scale, s, p, dp);
        }
        free(s);
        free(p);
        free(dp);
    }
    return failed ? -1 : 0;
}

/* The same from bf16 inputs (bit patterns, widened exactly to double). */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                    double *dq, double *dk, double *dv, double *delta, double *o, double *lse,
                    int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, int causal,
                    double scale, int nthreads) {
    if (!q || !k || !v || !dout || B < 0 || H < 0 || Nq < 1 || Nk < 1 || D < 1) return -1;
    const int64_t nq = B * H * Nq * D, nk = B * H * Nk * D;
    double *qd = (double *)malloc(sizeof(double) * (size_t)nq);
    double *dod = (double *)malloc(sizeof(double) * (size_t)nq);
    double *kd = (double *)malloc(sizeof(double) * (size_t)nk);
    double *vd = (double *)malloc(sizeof(double) * (size_t)nk);
    int rc = -1;
    if (qd && dod && kd && vd) {
        for (int64_t x = 0; x < nq; ++x) {
            qd[x] = widen_bf16_b(q[x]);
            dod[x] = widen_bf16_b(dout[x]);
        }
        for (int64_t x = 0; x < nk; ++x) {
            kd[x] = widen_bf16_b(k[x]);
            vd[x] = widen_bf16_b(v[x]);
        }
        rc = oracle_attn_bwd_f64(qd, kd, vd, dod, dq, dk, dv, delta, o, lse, B, H, Nq, Nk, D, causal,
                                 scale, nthreads);
    }
    free(qd);
    free(dod);
    free(kd);
    free(vd);
    return rc;
}

/* ------------------------------------------------------------------------
 * Sampled outputs of the same backward, for problems too large for the full
 * computation (each value is computed on its own, by the formulas above).
 */

/* Row statistics of query row i of one slice: visible keys n_vis, max m,
 * sum l (of exp(s - m)); s, scratch of Nk doubles, receives the scores. */
static int64_t row_scores(const double *qi, const double *kb, int64_t i, int64_t Nq, int64_t Nk, int64_t D,
                          int causal, double scale, double *s, double *m_out, double *l_out) {
    int64_t n_vis = Nk, j, d;
    if (causal) {
        n_vis = i + (Nk - Nq) + 1;
        if (n_vis > Nk) n_vis = Nk;
        if (n_vis < 0) n_vis = 0;
    }
    double m = -INFINITY, l = 0.0;
    for (j = 0; j < n_vis; ++j) {
        double a = 0.0;
        for (d = 0; d < D; ++d) a += qi[d] * kb[j * D + d];
        s[j] = scale * a;
        if (s[j] > m) m = s[j];
    }
    for (j = 0; j < n_vis; ++j) l += exp(s[j] - m);
    *m_out = m;
    *l_out = l;
    return n_vis;
}

static void widen_slice(const uint16_t *src, double *dst, int64_t n) {
    for (int64_t x = 0; x < n; ++x) dst[x] = widen_bf16_b(src[x]);
}

/* dQ and D for the rows (bh_idx[r], row_idx[r]): dq_out [R*D], delta_out [R].
 * Inputs as oracle_attn_bwd (bf16 bit patterns, [BH, N, D]). */
int oracle_attn_bwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                         int64_t BH, int64_t Nq, int64_t Nk, int64_t D, int causal, double scale,
                         const int64_t *bh_idx, const int64_t *row_idx, int64_t R, double *dq_out,
                         double *delta_out, int nthreads) {
    if (!q || !k || !v || !dout || !bh_idx || !row_idx || !dq_out || !delta_out) return -1;
    if (BH < 1 || Nq < 1 || Nk < 1 || D < 1 || R < 0) return -1;
    for (int64_t r = 0; r < R; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= Nq) return -1;
    int failed = 0;
    const int nt = nthreads_or_all(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt) reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *qi = (double *)malloc(sizeof(double) * (size_t)D);
        double *doi = (double *)malloc(sizeof(double) * (size_t)D);
        double *kj = (double *)malloc(sizeof(double) * (size_t)D);
        double *vj = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qi || !doi || !kj || !vj) {
            failed = 1;
        } else {
            int64_t r;
#pragma omp for schedule(dynamic, 1)
            for (r = 0; r < R; ++r) {
                const int64_t bh = bh_idx[r], i = row_idx[r];
                widen_slice(q + (bh * Nq + i) * D, qi, D);
                widen_slice(dout + (bh * Nq + i) * D, doi, D);
                const uint16_t *kb = k + bh * Nk * D, *vb = v + bh * Nk * D;
                double *dqr = dq_out + r * D;
                int64_t j, d;
                for (d = 0; d < D; ++d) dqr[d] = 0.0;
                int64_t n_vis = Nk;
                if (causal) {
                    n_vis = i + (Nk - Nq) + 1;
                    if (n_vis > Nk) n_vis = Nk;
                    if (n_vis < 0) n_vis = 0;
                }
                if (n_vis == 0) {
                    delta_out[r] = 0.0;
                    continue;
                }
                double m = -INFINITY, l = 0.0;
                for (j = 0; j < n_vis; ++j) {
                    widen_slice(kb + j * D, kj, D);
                    double a = 0.0;
                    for (d = 0; d < D; ++d) a += qi[d] * kj[d];
                    s[j] = scale * a;
                    if (s[j] > m) m = s[j];
                }
                for (j = 0; j < n_vis; ++j) l += exp(s[j] - m);
                /* D_i = sum_j p_ij dp_ij, then dq_i = scale sum_j p_ij (dp_ij - D_i) k_j */
                double dl = 0.0;
                for (j = 0; j < n_vis; ++j) {
                    widen_slice(vb + j * D, vj, D);
                    double a = 0.0;
                    for (d = 0; d < D; ++d) a += doi[d] * vj[d];
                    const double p = exp(s[j] - m) / l;
                    dl += p * a;
                    s[j] = a;  /* keep dp_ij; p is recomputed below from the stored max */
                }
                delta_out[r] = dl;
                /* second pass: recompute the scores for p (s now holds dp) */
                for (j = 0; j < n_vis; ++j) {
                    widen_slice(kb + j * D, kj, D);
                    double a = 0.0;
                    for (d = 0; d < D; ++d) a += qi[d] * kj[d];
                    const double p = exp(scale * a - m) / l;
                    const double ds = p * (s[j] - dl);
                    for (d = 0; d < D; ++d) dqr[d] += scale * ds * kj[d];
                }
            }
        }
        free(s);
        free(qi);
        free(doi);
        free(kj);
        free(vj);
    }
    return failed ? -1 : 0;
}

/* dK and dV for the keys key_idx[r] of slice bh: dk_out, dv_out [R*D].  The
 * slice's per-row max, sum and D are computed once (the whole slice's scores),
 * then each key's gradients from all the queries that see it. */
int oracle_attn_bwd_keys(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                         int64_t BH, int64_t Nq, int64_t Nk, int64_t D, int causal, double scale, int64_t bh,
                         const int64_t *key_idx, int64_t R, double *dk_out, double *dv_out, int nthreads) {
    if (!q || !k || !v || !dout || !key_idx || !dk_out || !dv_out) return -1;
    if (BH < 1 || Nq < 1 || Nk < 1 || D < 1 || R < 0 || bh < 0 || bh >= BH) return -1;
    for (int64_t r = 0; r < R; ++r)
        if (key_idx[r] < 0 || key_idx[r] >= Nk) return -1;
    double *qd = (double *)malloc(sizeof(double) * (size_t)(Nq * D));
    double *dod = (double *)malloc(sizeof(double) * (size_t)(Nq * D));
    double *kd = (double *)malloc(sizeof(double) * (size_t)(Nk * D));
    double *vd = (double *)malloc(sizeof(double) * (size_t)(Nk * D));
    double *mrow = (double *)malloc(sizeof(double) * (size_t)Nq);
    double *lrow = (double *)malloc(sizeof(double) * (size_t)Nq);
    double *drow = (double *)malloc(sizeof(double) * (size_t)Nq);
    int failed = !qd || !dod || !kd || !vd || !mrow || !lrow || !drow;
    const int nt = nthreads_or_all(nthreads);
    (void)nt;
    if (!failed) {
        widen_slice(q + bh * Nq * D, qd, Nq * D);
        widen_slice(dout + bh * Nq * D, dod, Nq * D);
        widen_slice(k + bh * Nk * D, kd, Nk * D);
        widen_slice(v + bh * Nk * D, vd, Nk * D);
#pragma omp parallel num_threads(nt) reduction(| : failed)
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
            if (!s) {
                failed = 1;
            } else {
                int64_t i;
#pragma omp for schedule(dynamic, 16)
                for (i = 0; i < Nq; ++i) {
                    double m, l;
                    const int64_t n_vis = row_scores(qd + i * D, kd, i, Nq, Nk, D, causal, scale, s, &m, &l);
                    mrow[i] = m;
                    lrow[i] = l;
                    double dl = 0.0;
                    for (int64_t j = 0; j < n_vis; ++j) {
                        double a = 0.0;
                        for (int64_t d = 0; d < D; ++d) a += dod[i * D + d] * vd[j * D + d];
                        dl += exp(s[j] - m) / l * a;
                    }
                    drow[i] = dl;
                }
            }
            free(s);
        }
    }
    if (!failed) {
        int64_t r;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
        for (r = 0; r < R; ++r) {
            const int64_t j = key_idx[r];
            double *dkr = dk_out + r * D, *dvr = dv_out + r * D;
            for (int64_t d = 0; d < D; ++d) {
                dkr[d] = 0.0;
                dvr[d] = 0.0;
            }
            /* queries that see key j: all, or i >= j - (Nk - Nq) when causal */
            int64_t i0 = 0;
            if (causal) {
                i0 = j - (Nk - Nq);
                if (i0 < 0) i0 = 0;
            }
            for (int64_t i = i0; i < Nq; ++i) {
                double a = 0.0, b = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    a += qd[i * D + d] * kd[j * D + d];
                    b += dod[i * D + d] * vd[j * D + d];
                }
                const double p = exp(scale * a - mrow[i]) / lrow[i];
                const double ds = p * (b - drow[i]);
                for (int64_t d = 0; d < D; ++d) {
                    dvr[d] += p * dod[i * D + d];
                    dkr[d] += scale * ds * qd[i * D + d];
                }
            }
        }
    }
    free(qd);
    free(dod);
    free(kd);
    free(vd);
    free(mrow);
    free(lrow);
    free(drow);
    return failed ? -1 : 0;
}
