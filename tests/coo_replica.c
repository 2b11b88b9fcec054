/*
 * coo_replica.c -- test checker: a CPU replica, in fp32, of the decision that
 * libsot's thresholded COO extraction takes for every pair ("From Theory to
 * Throughput: CUDA-Optimized APML", Abstract / Innovation: negligible
 * assignments are thresholded and the plan is stored in COO form,
 * bidirectionally).
 *
 * It is not the oracle.  The oracle decides in fp64 from the definition; this
 * file re-takes the library's own fp32 decisions, from the fp32 operands the
 * library reports (sot_plan_coo_operands), with the operation order that
 * include/sot.h documents for that call.  Every step is one IEEE-754 binary32
 * operation rounded to nearest even: a product, a sum, or fmaf (one rounding).
 * Compile without contraction (-ffp-contract=off) and without fast-math, so
 * that the compiler neither fuses nor reorders these steps.
 *
 * Given the operands, the support is a function of them alone, so the
 * library's index lists must equal this file's exactly, and its row and column
 * maxima must equal the maxima recomputed here bit for bit.
 */
#include <math.h>
#include <stdlib.h>

/* Score of one ordered pair in the point layout (d <= 3):
 *   -(base + sum_k fl(p_k + q_k)^2), each square added by fmaf, k ascending. */
static float point_score(int d, float base, const float *p, const float *q) {
    float acc = base;
    for (int k = 0; k < d; ++k) {
        const float t = p[k] + q[k];
        acc = fmaf(t, t, acc);
    }
    return -acc;
}

/* Dot product in the dense layout (d > 3): fmaf chain from 0, k ascending. */
static float dense_dot(int d, const float *x, const float *y) {
    float acc = 0.0f;
    for (int k = 0; k < d; ++k) acc = fmaf(x[k], y[k], acc);
    return acc;
}

/* Row score t_ij and column score t'_ij of pair (i, j). */
static void pair_scores(int d, const float *u, const float *nu, const float *v, const float *nv,
                        const float *xc, const float *yc, float two_kappa, float brow, float bcol,
                        float *t_row, float *t_col) {
    if (d <= 3) {
        *t_row = point_score(d, brow, u, nv);
        *t_col = point_score(d, bcol, v, nu);
    } else {
        const float p = dense_dot(d, xc, yc);
        *t_row = fmaf(two_kappa, p, -brow);
        *t_col = fmaf(two_kappa, p, -bcol);
    }
}

/*
 * One cloud.  Inputs as sot_plan_coo_operands writes them: xc[n][d], lwx[n],
 * Lx[n], yc[m][d], lwy[m], Ly[m], kappa, log2tau.  Outputs: Mr[n], Mc[m]
 * (the maxima recomputed here) and, when rows != NULL and cap is large
 * enough, the kept pairs in row-major order.  Returns the number of kept
 * pairs, or -1 on bad arguments, -2 when memory runs out.
 */
long long coo_replica(int n, int m, int d, const float *xc, const float *lwx, const float *Lx,
                      const float *yc, const float *lwy, const float *Ly, float kappa, float log2tau,
                      int dirs, float *Mr, float *Mc, long long cap, int *rows, int *cols) {
    if (n <= 0 || m <= 0 || d <= 0 || dirs < 1 || dirs > 3) return -1;
    const int dd = d <= 3 ? 3 : 1;
    /* point layout: u = fl(sqrt(kappa) x), nu = -u (exact); the same for y */
    float *u = (float *)calloc((size_t)n * dd, sizeof(float));
    float *nu = (float *)calloc((size_t)n * dd, sizeof(float));
    float *v = (float *)calloc((size_t)m * dd, sizeof(float));
    float *nv = (float *)calloc((size_t)m * dd, sizeof(float));
    float *brow = (float *)malloc(sizeof(float) * (size_t)m); /* fl(lwy_j - Ly_j) negated */
    float *bcol = (float *)malloc(sizeof(float) * (size_t)n); /* fl(lwx_i - Lx_i) negated */
    long long *cnt = (long long *)malloc(sizeof(long long) * ((size_t)n + 1));
    if (!u || !nu || !v || !nv || !brow || !bcol || !cnt) {
        free(u); free(nu); free(v); free(nv); free(brow); free(bcol); free(cnt);
        return -2;
    }
    const float sk = sqrtf(kappa);
    const float two_kappa = 2.0f * kappa;
    if (d <= 3) {
        for (int i = 0; i < n; ++i)
            for (int k = 0; k < d; ++k) {
                u[(size_t)i * 3 + k] = sk * xc[(size_t)i * d + k];
                nu[(size_t)i * 3 + k] = -u[(size_t)i * 3 + k];
            }
        for (int j = 0; j < m; ++j)
            for (int k = 0; k < d; ++k) {
                v[(size_t)j * 3 + k] = sk * yc[(size_t)j * d + k];
                nv[(size_t)j * 3 + k] = -v[(size_t)j * 3 + k];
            }
    }
    for (int j = 0; j < m; ++j) brow[j] = -(lwy[j] - Ly[j]);
    for (int i = 0; i < n; ++i) bcol[i] = -(lwx[i] - Lx[i]);

    /* maxima */
    for (int j = 0; j < m; ++j) Mc[j] = -INFINITY;
    for (int i = 0; i < n; ++i) {
        float mr = -INFINITY;
        for (int j = 0; j < m; ++j) {
            float tr, tc;
            pair_scores(d, u + (size_t)i * dd, nu + (size_t)i * dd, v + (size_t)j * dd, nv + (size_t)j * dd,
                        xc + (size_t)i * d, yc + (size_t)j * d, two_kappa, brow[j], bcol[i], &tr, &tc);
            mr = fmaxf(mr, tr);
            Mc[j] = fmaxf(Mc[j], tc);
        }
        Mr[i] = mr;
    }

    /* predicate: count per row, then the ordered write */
    for (int pass = 0; pass < 2; ++pass) {
        long long o = 0;
        cnt[0] = 0;
        for (int i = 0; i < n; ++i) {
            const float thr_r = Mr[i] + log2tau;
            for (int j = 0; j < m; ++j) {
                float tr, tc;
                pair_scores(d, u + (size_t)i * dd, nu + (size_t)i * dd, v + (size_t)j * dd,
                            nv + (size_t)j * dd, xc + (size_t)i * d, yc + (size_t)j * d, two_kappa, brow[j],
                            bcol[i], &tr, &tc);
                int keep = 0;
                if (dirs & 1) keep = tr >= thr_r;
                if (dirs & 2) keep = keep || (tc >= Mc[j] + log2tau);
                if (keep) {
                    if (pass == 1) {
                        rows[o] = i;
                        cols[o] = j;
                    }
                    ++o;
                }
            }
            cnt[i + 1] = o;
        }
        if (pass == 0 && (!rows || cap < o)) break;
    }
    const long long total = cnt[n];
    free(u); free(nu); free(v); free(nv); free(brow); free(bcol); free(cnt);
    return total;
}
