/*
 * CPU oracle for the Based linear-attention forward.  TEST INFRASTRUCTURE
 * ONLY: the tests, the package's smoke check and the bench's CPU-baseline leg
 * are its only callers.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * The pages name the kernel ("GPU의 폭발적인 성능 향상", news.hada.io topic
 * 14783, section "ThunderKittens"; "GPUの爆発的な性能向上", ja.news.hada.io,
 * section "FlashAttentionの例と性能": a Based linear-attention forward at
 * 215 TFLOP/s on an H100) but print no formula.  The definition used here is
 * the one published with Based (Arora et al., 2024, "Simple linear attention
 * language models balance the recall-throughput tradeoff"): causal linear
 * attention whose kernel is the second-order Taylor polynomial of exp,
 *
 *   s_ij = scale * sum_a q_ia k_ja            (feature dim F, scale = 1/sqrt(F))
 *   a_ij = 1 + s_ij + s_ij^2 / 2              (j <= i; a_ij >= 1/2 > 0)
 *   z_i  = sum_{j <= i} a_ij
 *   y_id = sum_{j <= i} a_ij v_jd / z_i
 *
 * which is what the feature map phi(x) = [1, x, vec(x x^T)/sqrt(2)] (scaled)
 * gives as phi(q_i) . phi(k_j); linear attention reaches the same numbers
 * through a running sum of phi(k_j) v_j^T, in any order of rounding.  This
 * oracle is the plain quadratic definition, in fp64, from the same bf16 bytes
 * the GPU reads (each widens to double exactly), in the order above; every sum
 * runs in increasing index order.  Rows are independent and spread over OpenMP
 * threads, which changes no result.
 *
 * Layout: q, k [B*H, N, F]; v, y [B*H, N, D]; z [B*H, N]; row-major, the last
 * dimension innermost.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double based_widen(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One output row (bh, i): y_row[D] and *z_out. qd: scratch of F doubles. */
static void based_row(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t N, int64_t F,
                      int64_t D, double scale, int64_t bh, int64_t i, double *qd, double *y_row,
                      double *z_out) {
    const uint16_t *qi = q + (bh * N + i) * F;
    const uint16_t *kb = k + bh * N * F;
    const uint16_t *vb = v + bh * N * D;
    int64_t j, a, d;
    for (a = 0; a < F; ++a) qd[a] = based_widen(qi[a]);
    for (d = 0; d < D; ++d) y_row[d] = 0.0;
    double z = 0.0;
    for (j = 0; j <= i; ++j) {
        const uint16_t *kj = kb + j * F;
        double dot = 0.0;
        for (a = 0; a < F; ++a) dot += qd[a] * based_widen(kj[a]);
        const double s = scale * dot;
        const double w = 1.0 + s + 0.5 * s * s;
        z += w;
        const uint16_t *vj = vb + j * D;
        for (d = 0; d < D; ++d) y_row[d] += w * based_widen(vj[d]);
    }
    for (d = 0; d < D; ++d) y_row[d] /= z;
    *z_out = z;
}

static int based_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* The whole problem: y [BH, N, D], z [BH, N].  Returns 0, or -1 on bad sizes. */
int oracle_based_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *y, double *z,
                     int64_t BH, int64_t N, int64_t F, int64_t D, double scale, int nthreads) {
    if (BH < 0 || N < 0 || F < 1 || D < 1) return -1;
    const int64_t rows = BH * N;
    int bad = 0;
#pragma omp parallel num_threads(based_threads(nthreads)) reduction(| : bad)
    {
        double *qd = (double *)malloc(sizeof(double) * (size_t)F);
        if (!qd) {
            bad = 1;
        } else {
            int64_t r;
#pragma omp for schedule(dynamic, 16)
            for (r = 0; r < rows; ++r) {
                const int64_t bh = r / N, i = r % N;
                based_row(q, k, v, N, F, D, scale, bh, i, qd, y + r * D, z + r);
            }
            free(qd);
        }
    }
    return bad ? -1 : 0;
}

/* Sampled rows (bh_idx[t], row_idx[t]) only: y [R, D], z [R]. */
int oracle_based_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t BH, int64_t N,
                      int64_t F, int64_t D, double scale, const int64_t *bh_idx, const int64_t *row_idx,
                      int64_t R, double *y, double *z, int nthreads) {
    int64_t t;
    for (t = 0; t < R; ++t)
        if (bh_idx[t] < 0 || bh_idx[t] >= BH || row_idx[t] < 0 || row_idx[t] >= N) return -1;
    int bad = 0;
#pragma omp parallel num_threads(based_threads(nthreads)) reduction(| : bad)
    {
        double *qd = (double *)malloc(sizeof(double) * (size_t)F);
        if (!qd) {
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (t = 0; t < R; ++t) based_row(q, k, v, N, F, D, scale, bh_idx[t], row_idx[t], qd, y + t * D, z + t);
            free(qd);
        }
    }
    return bad ? -1 : 0;
}
