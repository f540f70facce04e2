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
