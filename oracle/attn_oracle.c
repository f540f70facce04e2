/*
 * CPU oracle for the attention forward.  TEST INFRASTRUCTURE ONLY: the tests,
 * the package's smoke check and the bench's CPU-baseline leg are its only
 * callers.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of attention, in fp64, from the
 * same bf16 bytes the GPU reads (each bf16 value widens to double exactly):
 *
 *   - "[GPU] Deep Learning for HPC" (bkkhyunn.github.io, hardware/pytorch_for_HPC),
 *     section "Flash Attention": the score matrix is Q times K-transpose, a
 *     softmax is applied to it, and the result multiplies V.  FlashAttention
 *     reaches the same result tile by tile; only the order of rounding differs.
 *   - null-ptr.tistory.com, category "development", the softmax post
 *     ("Original softmax"): sigma_i(z) = e^{z_i} / sum_j e^{z_j}, made safe
 *     against overflow by subtracting the row maximum first.
 *   - same site, the Triton `_fwd_kernel` post: the forward takes a
 *     `softmax_scale`, an `IS_CAUSAL` flag and returns `Lse` next to `Out`.
 *
 * Readings where the pages are silent (each listed with its reason in the
 * design notes): the scale multiplies the logits before the max and the exp;
 * causal means key j is visible to query i iff j <= i + (Nk - Nq) (aligned at
 * the bottom-right corner of the score matrix, which for Nq = Nk is j <= i);
 * LSE is the natural log of sum_j exp(s_ij) over visible keys, i.e.
 * m_i + log(l_i); layout is [B, H, Nq, D] for Q and O, [B, H, Nk, D] for K and
 * V, row-major with D innermost.
 *
 * Per output row (b, h, i), in this order:
 *   1. s_ij = scale * sum_d q_id k_jd           for every visible key j
 *   2. m_i  = max_j s_ij;  l_i = sum_j exp(s_ij - m_i)          (pass 1)
 *   3. p_ij = exp(s_ij - m_i) / l_i;  o_id = sum_j p_ij v_jd    (pass 2)
 *   4. lse_i = m_i + log(l_i)
 * Every sum runs in increasing index order in double precision.  Rows are
 * independent and are spread over OpenMP threads; that changes no result.
 * A row with no visible key (only when causal and Nq > Nk, for the first
 * Nq - Nk queries) gives o = 0 and lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One output row.  s: scratch of Nk doubles; qd: scratch of D doubles; p_row:
 * optional Nk doubles that receive p_ij (zero for invisible keys). */
static void attn_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t Nq, int64_t Nk, int64_t D, int causal, double scale,
                     int64_t bh, int64_t i, double *s, double *qd,
                     double *o_row, double *lse_out, double *p_row) {
    const uint16_t *qi = q + (bh * Nq + i) * D;
    const uint16_t *kb = k + bh * Nk * D;
    const uint16_t *vb = v + bh * Nk * D;
    int64_t n_vis = Nk;
    if (causal) {
        n_vis = i + (Nk - Nq) + 1; /* keys 0 .. i + Nk - Nq */
        if (n_vis > Nk) n_vis = Nk;
        if (n_vis < 0) n_vis = 0;
    }
    int64_t j, d;

    for (d = 0; d < D; ++d) qd[d] = widen_bf16(qi[d]);

    /* step 1: scaled scores; four keys at a time only for instruction-level
     * parallelism -- each dot product is still summed in index order. */
    for (j = 0; j + 4 <= n_vis; j += 4) {
        const uint16_t *k0 = kb + (j + 0) * D, *k1 = kb + (j + 1) * D;
        const uint16_t *k2 = kb + (j + 2) * D, *k3 = kb + (j + 3) * D;
        double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
        for (d = 0; d < D; ++d) {
            a0 += qd[d] * widen_bf16(k0[d]);
            a1 += qd[d] * widen_bf16(k1[d]);
            a2 += qd[d] * widen_bf16(k2[d]);
            a3 += qd[d] * widen_bf16(k3[d]);
        }
        s[j + 0] = scale * a0;
        s[j + 1] = scale * a1;
        s[j + 2] = scale * a2;
        s[j + 3] = scale * a3;
    }
    for (; j < n_vis; ++j) {
        const uint16_t *kj = kb + j * D;
        double a = 0.0;
        for (d = 0; d < D; ++d) a += qd[d] * widen_bf16(kj[d]);
        s[j] = scale * a;
    }

    for (d = 0; d < D; ++d) o_row[d] = 0.0;
    if (p_row)
        for (j = 0; j < Nk; ++j) p_row[j] = 0.0;
    if (n_vis <= 0) {
        *lse_out = -INFINITY;
        return;
    }

    /* step 2: safe softmax, pass 1 */
    double m = s[0];
    for (j = 1; j < n_vis; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (j = 0; j < n_vis; ++j) l += exp(s[j] - m);

    /* step 3: pass 2 -- normalised probabilities times V */
    for (j = 0; j < n_vis; ++j) {
        const double p = exp(s[j] - m) / l;
        const uint16_t *vj = vb + j * D;
        if (p_row) p_row[j] = p;
        for (d = 0; d < D; ++d) o_row[d] += p * widen_bf16(vj[d]);
    }

    /* step 4 */
    *lse_out = m + log(l);
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of OpenMP threads a call with `nthreads` would use (0 = all). */
int oracle_threads(int nthreads) { return set_threads(nthreads); }

/* Whole forward: q, o [B*H*Nq*D], k, v [B*H*Nk*D], lse [B*H*Nq], fp64.
 * Returns 0, or -1 on a bad argument or a failed scratch allocation. */
int oracle_attn_fwd_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       double *o, double *lse, int64_t B, int64_t H, int64_t Nq,
                       int64_t Nk, int64_t D, int causal, double scale, int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 0 || H < 0 || Nq < 0 || Nk < 0 || D < 1) return -1;
    const int64_t rows = B * H * Nq;
    int failed = 0;
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt) reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd) {
            failed = 1;
        } else {
            int64_t r;
#pragma omp for schedule(dynamic, 16)
            for (r = 0; r < rows; ++r) {
                attn_row(q, k, v, Nq, Nk, D, causal, scale, r / Nq, r % Nq, s, qd,
                         o + r * D, lse + r, NULL);
            }
        }
        free(s);
        free(qd);
    }
    return failed ? -1 : 0;
}

/* Square case (Nq = Nk = N): o [B*H*N*D] and lse [B*H*N]. */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    double *o, double *lse, int64_t B, int64_t H, int64_t N,
                    int64_t D, int causal, double scale, int nthreads) {
    return oracle_attn_fwd_qk(q, k, v, o, lse, B, H, N, N, D, causal, scale, nthreads);
}

/* Selected rows only: row r is query (bh_idx[r], row_idx[r]); o [nrows*D], lse [nrows]. */
int oracle_attn_rows_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        int64_t BH, int64_t Nq, int64_t Nk, int64_t D, int causal, double scale,
                        const int64_t *bh_idx, const int64_t *row_idx, int64_t nrows,
                        double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || !bh_idx || !row_idx || Nq < 1 || Nk < 1 || D < 1) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= Nq) return -1;
    int failed = 0;
    const int nt = set_threads(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt) reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd) {
            failed = 1;
        } else {
            int64_t r;
#pragma omp for schedule(dynamic, 4)
            for (r = 0; r < nrows; ++r)
                attn_row(q, k, v, Nq, Nk, D, causal, scale, bh_idx[r], row_idx[r], s, qd,
                         o + r * D, lse + r, NULL);
        }
        free(s);
        free(qd);
    }
    return failed ? -1 : 0;
}

/* Square case of oracle_attn_rows_qk. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t BH, int64_t N, int64_t D, int causal, double scale,
                     const int64_t *bh_idx, const int64_t *row_idx, int64_t nrows,
                     double *o, double *lse, int nthreads) {
    return oracle_attn_rows_qk(q, k, v, BH, N, N, D, causal, scale, bh_idx, row_idx, nrows, o, lse,
                               nthreads);
}

/* The probability matrix as well (small problems): p [B*H*Nq*Nk], o, lse as above. */
int oracle_attn_probs_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         double *o, double *lse, double *p, int64_t B, int64_t H,
                         int64_t Nq, int64_t Nk, int64_t D, int causal, double scale) {
    if (!q || !k || !v || !o || !lse || !p || B < 0 || H < 0 || Nq < 1 || Nk < 1 || D < 1) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !qd) {
        free(s);
        free(qd);
        return -1;
    }
    for (int64_t r = 0; r < B * H * Nq; ++r)
        attn_row(q, k, v, Nq, Nk, D, causal, scale, r / Nq, r % Nq, s, qd, o + r * D, lse + r,
                 p + r * Nk);
    free(s);
    free(qd);
    return 0;
}

/* Square case of oracle_attn_probs_qk. */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      double *o, double *lse, double *p, int64_t B, int64_t H,
                      int64_t N, int64_t D, int causal, double scale) {
    return oracle_attn_probs_qk(q, k, v, o, lse, p, B, H, N, N, D, causal, scale);
}
