/*
 * oracle.c -- plain, slow, fp64 CPU reference for log-domain Sinkhorn between
 * point clouds with squared-Euclidean cost.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline of the benchmark load this library.  It shares no code, header,
 * table or helper with the CUDA library; the two meet only through the seeded
 * input arrays.
 *
 * What it follows (page titles and sections):
 *   - "FlashSinkhorn: IO-aware entropic optimal transport on GPU",
 *     Methodologie 1 (Propositie 1): the stabilised log-domain update
 *         f_i <- -eps * LSE_j[ (g_j - C_ij)/eps + log b_j ]
 *     and its mirror for g.  This file evaluates exactly that expression,
 *     with C_ij = sum_k (x_ik - y_jk)^2 in the direct (difference) form and a
 *     two-pass log-sum-exp (max first, then the sum of exp(v - max)).
 *   - same page, Methodologie 2 ("Online LSE"): the LSE is exact, so a
 *     two-pass LSE is the reference for it.
 *   - same page, Methodologie 3 ("transport matrix application"): the plan
 *     P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps) applied to Y gives the
 *     gradient 2(a_i x_i - sum_j P_ij y_j) and the cost sum_ij P_ij C_ij;
 *     applied to any matrix V it gives the transport-matrix products
 *     P V and P^T U that the page's streaming HVP is built from; the HVP
 *     itself (orc_hvp) is the Hessian of the converged loss with respect to
 *     X applied to V, by implicit differentiation of the marginal conditions
 *     (the page gives no formula: this is the plain reading).
 *   - "From Theory to Throughput: CUDA-Optimized APML", Abstract and
 *     Innovation: negligible assignments are thresholded, the plan is kept in
 *     COO form with bidirectional symmetrisation, gradients are kept on the
 *     stored support; on that support the loss runs an adaptive softmax,
 *     bidirectional symmetrisation and Sinkhorn normalisation (orc_apml_coo;
 *     the page does not give the temperature: the caller passes it).
 *
 * Readings where the pages are silent (each one listed in the design notes):
 *   - one iteration = f-half then g-half using the new f (Gauss-Seidel), from
 *     f = g = 0 unless warm-started;
 *   - eps annealing eps_k = max(eps_min, eps0 * factor^k), a fixed number of
 *     iterations per stage, a marginal-error stop test applied at the final
 *     eps (or at every stage with early exit);
 *   - marginal error = sum_i | sum_j P_ij - a_i |;
 *   - COO support = { P_ij >= tau * max_j' P_ij' } U { P_ij >= tau * max_i' P_i'j },
 *     row-major order;
 *   - cosine cost ("FlashSinkhorn", Conclusies: the structure also holds for
 *     the cosine distance after normalisation): C_ij = 2 - 2 x_i.y_j / (|x_i| |y_j|)
 *     for nonzero points.  A zero point has no direction: it normalises to the
 *     zero vector, so C_ij = [x_i != 0] + [y_j != 0] - 2 xhat_i.yhat_j in general.
 *
 * Parity pins (tests, CPU only): closed forms at n = m = 1 and for 2 x 2
 * problems, the attention-form identity, marginals and duality at
 * convergence, brute-force assignment on tiny clouds, the d = 1 sorted
 * matching, the large-eps closed form, translation / rotation / swap
 * invariances, shift invariance, finite differences of the dual objective,
 * and for the HVP finite differences of the gradient, second differences of
 * the dual, symmetry and the n = 1 and large-eps limits.
 *
 * Compile: cc -O2 -fopenmp -fPIC -shared oracle.c -lm  (no fast-math).
 * Optional -DORC_MUTANT=k builds a deliberately wrong variant (k = 1..14) that
 * the test suite uses to show that the pins catch plausible mistakes.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

int orc_mutant(void) { return ORC_MUTANT; }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* Cost selected for every call that follows: 0 squared Euclidean, 1 cosine. */
static int g_cost = 0;
void orc_set_cost(int kind) { g_cost = (kind == 1) ? 1 : 0; }
int orc_get_cost(void) { return g_cost; }

static double norm2(const double *v, int d) {
    double s = 0.0;
    for (int k = 0; k < d; ++k) s += v[k] * v[k];
    return sqrt(s);
}

/* Cosine cost 2 - 2 cos(x, y) (zero points: see the header). */
static double cosine_ij(const double *x, const double *y, int d) {
    const double nx = norm2(x, d), ny = norm2(y, d);
    double dot = 0.0;
    for (int k = 0; k < d; ++k) dot += x[k] * y[k];
    double cs = 0.0;
    if (nx > 0.0 && ny > 0.0) {
#if ORC_MUTANT == 9
        cs = dot / nx; /* mutant: y not normalised */
#else
        cs = dot / (nx * ny);
#endif
    }
    return (nx > 0.0 ? 1.0 : 0.0) + (ny > 0.0 ? 1.0 : 0.0) - 2.0 * cs;
}

/* Squared Euclidean distance, direct form (or the cosine cost when selected). */
static double cost_ij(const double *x, const double *y, int d) {
    if (g_cost == 1) return cosine_ij(x, y, d);
    double c = 0.0;
#if ORC_MUTANT == 8
    d = d > 1 ? d - 1 : d; /* mutant: drops the last coordinate */
#endif
    for (int k = 0; k < d; ++k) {
        double t = x[k] - y[k];
        c += t * t;
    }
    return c;
}

/* Two-pass log-sum-exp: max first, then sum of exp(v - max). */
static double lse2(const double *v, int len) {
    double mx = -INFINITY;
    for (int k = 0; k < len; ++k)
        if (v[k] > mx) mx = v[k];
    if (mx == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int k = 0; k < len; ++k) s += exp(v[k] - mx);
#if ORC_MUTANT == 7
    return log(s); /* mutant: forgets to add the max back */
#else
    return mx + log(s);
#endif
}

/* f-half: f_i = -eps * LSE_j[(g_j - C_ij)/eps + log b_j]. */
int orc_f_half(int n, int m, int d, const double *X, const double *Y,
               const double *b, const double *g, double eps, double *f_out) {
    if (n <= 0 || m <= 0 || d <= 0 || !(eps > 0)) return -1;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)m);
        if (!s) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(static)
        for (int i = 0; i < n; ++i) {
            if (!s) continue;
            for (int j = 0; j < m; ++j) {
                double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
#if ORC_MUTANT == 1
                s[j] = (g[j] - c) / eps; /* mutant: drops log b_j */
#elif ORC_MUTANT == 2
                s[j] = (g[j] + c) / eps + log(b[j]); /* mutant: wrong sign of C */
#else
                s[j] = (g[j] - c) / eps + log(b[j]);
#endif
            }
            f_out[i] = -eps * lse2(s, m);
        }
        free(s);
    }
    return err;
}

/* g-half: g_j = -eps * LSE_i[(f_i - C_ij)/eps + log a_i]. */
int orc_g_half(int n, int m, int d, const double *X, const double *Y,
               const double *a, const double *b, const double *f, double eps,
               double *g_out) {
    if (n <= 0 || m <= 0 || d <= 0 || !(eps > 0)) return -1;
    (void)b;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        if (!s) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(static)
        for (int j = 0; j < m; ++j) {
            if (!s) continue;
            for (int i = 0; i < n; ++i) {
                double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
#if ORC_MUTANT == 3
                /* mutant: weights transposed (uses b where a belongs) */
                s[i] = (f[i] - c) / eps + log(b[i < m ? i : m - 1]);
#else
                s[i] = (f[i] - c) / eps + log(a[i]);
#endif
            }
            g_out[j] = -eps * lse2(s, n);
        }
        free(s);
    }
    return err;
}

/* Row sums r_i = sum_j P_ij of the plan given by (f, g) at eps. */
static int row_sums(int n, int m, int d, const double *X, const double *Y,
                    const double *a, const double *b, const double *f,
                    const double *g, double eps, double *r) {
    /* log b_j once per column (the same values the sum would compute per pair) */
    double *lb = (double *)malloc(sizeof(double) * (size_t)m);
    if (!lb) return -2;
    for (int j = 0; j < m; ++j) lb[j] = log(b[j]);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < n; ++i) {
        const double la = log(a[i]);
        double acc = 0.0;
        for (int j = 0; j < m; ++j) {
            double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
            acc += exp((f[i] + g[j] - c) / eps + la + lb[j]);
        }
        r[i] = acc;
    }
    free(lb);
    return 0;
}

/* Marginal L1 error of the row constraint: sum_i | sum_j P_ij - a_i |. */
double orc_marginal_err(int n, int m, int d, const double *X, const double *Y,
                        const double *a, const double *b, const double *f,
                        const double *g, double eps) {
    double *r = (double *)malloc(sizeof(double) * (size_t)n);
    if (!r) return NAN;
    if (row_sums(n, m, d, X, Y, a, b, f, g, eps, r)) {
        free(r);
        return NAN;
    }
    double e = 0.0;
    for (int i = 0; i < n; ++i) e += fabs(r[i] - a[i]);
    free(r);
    return e;
}

/* One full iteration: f-half, then g-half with the new f. */
static int iterate(int n, int m, int d, const double *X, const double *Y,
                   const double *a, const double *b, double eps, double *f,
                   double *g) {
#if ORC_MUTANT == 6
    /* mutant: Jacobi order -- the g-half sees the f from before this f-half */
    double *fold = (double *)malloc(sizeof(double) * (size_t)n);
    if (!fold) return -2;
    memcpy(fold, f, sizeof(double) * (size_t)n);
    int e = orc_f_half(n, m, d, X, Y, b, g, eps, f);
    if (!e) e = orc_g_half(n, m, d, X, Y, a, b, fold, eps, g);
    free(fold);
    return e;
#else
    int e = orc_f_half(n, m, d, X, Y, b, g, eps, f);
    if (e) return e;
    return orc_g_half(n, m, d, X, Y, a, b, f, eps, g);
#endif
}

/*
 * Fixed schedule: stage k runs iters[k] iterations at eps_list[k].
 * warm != 0 starts from the given f, g; otherwise from f = g = 0.
 */
int orc_sinkhorn(int n, int m, int d, const double *X, const double *Y,
                 const double *a, const double *b, int nstages,
                 const double *eps_list, const int *iters, double *f, double *g,
                 int warm) {
    if (n <= 0 || m <= 0 || d <= 0 || nstages < 0) return -1;
    if (!warm) {
        for (int i = 0; i < n; ++i) f[i] = 0.0;
        for (int j = 0; j < m; ++j) g[j] = 0.0;
    }
    for (int k = 0; k < nstages; ++k) {
        if (!(eps_list[k] > 0) || iters[k] < 0) return -1;
        for (int t = 0; t < iters[k]; ++t) {
            int e = iterate(n, m, d, X, Y, a, b, eps_list[k], f, g);
            if (e) return e;
        }
    }
    return 0;
}

/*
 * Number of annealing stages: eps_k = max(eps_min, eps0 * factor^k) for
 * k = 0, 1, ...; the first k with eps0 * factor^k <= eps_min is the last
 * (clamped) stage.  eps_out (if non-NULL, capacity cap) receives the values.
 */
int orc_anneal_stages(double eps0, double factor, double eps_min, double *eps_out,
                      int cap) {
    if (!(eps0 > 0) || !(eps_min > 0) || !(factor > 0) || !(factor < 1)) return -1;
    int k = 0;
    double e = eps0;
    for (;;) {
        double ek = e > eps_min ? e : eps_min;
        if (eps_out && k < cap) eps_out[k] = ek;
        ++k;
        if (e <= eps_min) break;
        e *= factor;
        if (k > 100000) return -1;
    }
    return k;
}

/*
 * Annealed solve with the marginal-error stop test.
 *   stages: orc_anneal_stages(eps0, factor, eps_min); iters_per_stage each.
 *   stop test err(f, g) < tol after an iteration, at the final eps only, or at
 *   every stage when early_exit != 0 (a passing test ends that stage).
 *   The final stage continues past iters_per_stage until the test passes or
 *   the total reaches max_iters.  No stage runs once max_iters is reached.
 * Outputs: f, g; stage_iters[k] realised per stage (capacity stage_cap);
 * *nstages_out, *iters_done, *err_out (err of the returned iterate, or NaN if
 * never evaluated), *converged.
 */
int orc_sinkhorn_anneal(int n, int m, int d, const double *X, const double *Y,
                        const double *a, const double *b, double eps0,
                        double factor, double eps_min, int iters_per_stage,
                        double tol, int max_iters, int early_exit, double *f,
                        double *g, int warm, int *stage_iters, int stage_cap,
                        int *nstages_out, int *iters_done, double *err_out,
                        int *converged) {
    int K = orc_anneal_stages(eps0, factor, eps_min, NULL, 0);
    if (K <= 0 || iters_per_stage < 0 || max_iters < 0) return -1;
    double *eps_list = (double *)malloc(sizeof(double) * (size_t)K);
    if (!eps_list) return -2;
    orc_anneal_stages(eps0, factor, eps_min, eps_list, K);
    if (!warm) {
        for (int i = 0; i < n; ++i) f[i] = 0.0;
        for (int j = 0; j < m; ++j) g[j] = 0.0;
    }
    int total = 0, conv = 0;
    double err = NAN;
    int k;
    for (k = 0; k < K; ++k) {
        int final_stage = (k == K - 1);
        int test = early_exit || final_stage;
        int done_here = 0;
        for (;;) {
            if (total >= max_iters) break;
            if (!final_stage && done_here >= iters_per_stage) break;
            if (final_stage && done_here >= iters_per_stage && !test) break;
            int e = iterate(n, m, d, X, Y, a, b, eps_list[k], f, g);
            if (e) { free(eps_list); return e; }
            ++total;
            ++done_here;
            if (test) {
                err = orc_marginal_err(n, m, d, X, Y, a, b, f, g, eps_list[k]);
                if (err < tol) {
                    if (final_stage) conv = 1;
                    break;
                }
            }
        }
        if (k < stage_cap && stage_iters) stage_iters[k] = done_here;
        if (conv || total >= max_iters) { ++k; break; }
    }
    if (nstages_out) *nstages_out = k;
    if (iters_done) *iters_done = total;
    if (err_out) *err_out = err;
    if (converged) *converged = conv;
    free(eps_list);
    return 0;
}

/*
 * Plan application with the final (f, g) at eps:
 *   P_ij = exp((f_i + g_j - C_ij)/eps + log a_i + log b_j)
 *   cost  = sum_ij P_ij C_ij
 *   grad  = 2 (a_i x_i - sum_j P_ij y_j)        [n x d]
 *           (cosine cost: sum_j P_ij dC_ij/dx_i with
 *            dC_ij/dx_i = -2 (yhat_j - (xhat_i.yhat_j) xhat_i) / |x_i|, 0 for a zero x_i)
 *   rowsum[i] = sum_j P_ij, colsum[j] = sum_i P_ij   (optional, may be NULL)
 */
int orc_plan_apply(int n, int m, int d, const double *X, const double *Y,
                   const double *a, const double *b, const double *f,
                   const double *g, double eps, double *cost, double *grad,
                   double *rowsum, double *colsum) {
    if (n <= 0 || m <= 0 || d <= 0 || !(eps > 0)) return -1;
    double total = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : total)
    for (int i = 0; i < n; ++i) {
        const double *xi = X + (size_t)i * d;
        double r = 0.0, q = 0.0;
        double *gi = grad ? grad + (size_t)i * d : NULL;
        if (gi)
            for (int k = 0; k < d; ++k) gi[k] = 0.0;
        const double nxi = norm2(xi, d);
        for (int j = 0; j < m; ++j) {
            const double *yj = Y + (size_t)j * d;
            double c = cost_ij(xi, yj, d);
#if ORC_MUTANT == 5
            double p = exp((f[i] - g[j] - c) / eps + log(a[i]) + log(b[j])); /* mutant: sign of g */
#else
            double p = exp((f[i] + g[j] - c) / eps + log(a[i]) + log(b[j]));
#endif
            r += p;
            q += p * c;
            if (gi && g_cost == 1) {
                const double nyj = norm2(yj, d);
                if (nxi > 0.0 && nyj > 0.0) {
                    double cs = 0.0;
                    for (int k = 0; k < d; ++k) cs += (xi[k] / nxi) * (yj[k] / nyj);
                    for (int k = 0; k < d; ++k) gi[k] += p * (-2.0) * (yj[k] / nyj - cs * xi[k] / nxi) / nxi;
                }
            } else if (gi) {
                for (int k = 0; k < d; ++k) gi[k] += p * yj[k];
            }
        }
        if (gi && g_cost != 1)
            for (int k = 0; k < d; ++k)
#if ORC_MUTANT == 4
                gi[k] = 2.0 * (xi[k] - gi[k]); /* mutant: drops a_i */
#else
                gi[k] = 2.0 * (a[i] * xi[k] - gi[k]);
#endif
        if (rowsum) rowsum[i] = r;
        total += q;
    }
    if (cost) *cost = total;
    if (colsum) {
#pragma omp parallel for schedule(static)
        for (int j = 0; j < m; ++j) {
            double s = 0.0;
            for (int i = 0; i < n; ++i) {
                double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
                s += exp((f[i] + g[j] - c) / eps + log(a[i]) + log(b[j]));
            }
            colsum[j] = s;
        }
    }
    return 0;
}

/*
 * Transport-matrix products ("FlashSinkhorn", Methodologie 3 and its HVP
 * paragraph), by the definition of P:
 *   side 0: out[i][:] = sum_j P_ij V[j][:]   (V is m x c, out is n x c)
 *   side 1: out[j][:] = sum_i P_ij V[i][:]   (V is n x c, out is m x c)
 */
int orc_transport(int n, int m, int d, const double *X, const double *Y,
                  const double *a, const double *b, const double *f,
                  const double *g, double eps, const double *V, int c,
                  int side, double *out) {
    if (n <= 0 || m <= 0 || d <= 0 || c <= 0 || !(eps > 0) || (side != 0 && side != 1)) return -1;
    const int nout = side == 0 ? n : m;
#pragma omp parallel for schedule(static)
    for (int o = 0; o < nout; ++o) {
        double *acc = out + (size_t)o * c;
        for (int k = 0; k < c; ++k) acc[k] = 0.0;
        const int nin = side == 0 ? m : n;
        for (int q = 0; q < nin; ++q) {
            const int i = side == 0 ? o : q, j = side == 0 ? q : o;
            const double cij = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
#if ORC_MUTANT == 10
            const double p = exp((f[i] + g[j] - cij) / eps + log(a[j % n]) + log(b[j])); /* mutant: wrong row weight */
#else
            const double p = exp((f[i] + g[j] - cij) / eps + log(a[i]) + log(b[j]));
#endif
            const double *v = V + (size_t)q * c;
            for (int k = 0; k < c; ++k) acc[k] += p * v[k];
        }
    }
    return 0;
}

/*
 * Objectives for the duality check:
 *   dual   = <a, f> + <b, g>
 *   primal = <C, P> + eps * KL(P || a x b),  KL(p||q) = sum p log(p/q) - p + q,
 * with log P_ij taken from P itself (not from the potentials formula).
 */
int orc_objectives(int n, int m, int d, const double *X, const double *Y,
                   const double *a, const double *b, const double *f,
                   const double *g, double eps, double *dual, double *primal) {
    double du = 0.0;
    for (int i = 0; i < n; ++i) du += a[i] * f[i];
    for (int j = 0; j < m; ++j) du += b[j] * g[j];
    double pr = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : pr)
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < m; ++j) {
            double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
            double q = a[i] * b[j];
            double p = exp((f[i] + g[j] - c) / eps + log(a[i]) + log(b[j]));
            double kl = (p > 0 ? p * log(p / q) : 0.0) - p + q;
            pr += p * c + eps * kl;
        }
    }
    *dual = du;
    *primal = pr;
    return 0;
}

/*
 * Row and column maxima of the log-domain scores:
 *   Mr_i = max_j [(g_j - C_ij)/eps + log b_j]
 *   Mc_j = max_i [(f_i - C_ij)/eps + log a_i]
 */
int orc_maxima(int n, int m, int d, const double *X, const double *Y,
               const double *a, const double *b, const double *f,
               const double *g, double eps, double *Mr, double *Mc) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < n; ++i) {
        double mx = -INFINITY;
        for (int j = 0; j < m; ++j) {
            double s = (g[j] - cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d)) / eps + log(b[j]);
            if (s > mx) mx = s;
        }
        Mr[i] = mx;
    }
#pragma omp parallel for schedule(static)
    for (int j = 0; j < m; ++j) {
        double mx = -INFINITY;
        for (int i = 0; i < n; ++i) {
            double s = (f[i] - cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d)) / eps + log(a[i]);
            if (s > mx) mx = s;
        }
        Mc[j] = mx;
    }
    return 0;
}

/*
 * Thresholded COO support in row-major order.  For each pair the margin is
 *   mu_ij = max( s_ij - (Mr_i + log tau),  s'_ij - (Mc_j + log tau) )
 * (row test, column test; dirs bit 1 = row test, bit 2 = column test), with
 * s_ij = (g_j - C_ij)/eps + log b_j and s'_ij = (f_i - C_ij)/eps + log a_i.
 * The support is mu_ij >= 0.  This routine lists every pair with
 * mu_ij >= -band (band >= 0), so a caller can separate the pairs that are
 * decided with room to spare from those near the threshold.
 * tau = 0 gives the full dense support (log 0 = -inf).
 * Returns the number of listed pairs; writes at most cap of them.
 */
long long orc_coo(int n, int m, int d, const double *X, const double *Y,
                  const double *a, const double *b, const double *f,
                  const double *g, double eps, double tau, int dirs, double band,
                  long long cap, int *rows, int *cols, double *vals,
                  double *margins) {
    if (!(tau >= 0) || dirs < 1 || dirs > 3 || !(band >= 0)) return -1;
    double *Mr = (double *)malloc(sizeof(double) * (size_t)n);
    double *Mc = (double *)malloc(sizeof(double) * (size_t)m);
    long long *cnt = (long long *)malloc(sizeof(long long) * (size_t)(n + 1));
    if (!Mr || !Mc || !cnt) { free(Mr); free(Mc); free(cnt); return -2; }
    orc_maxima(n, m, d, X, Y, a, b, f, g, eps, Mr, Mc);
#if ORC_MUTANT == 13
    double lt = tau > 0 ? -log(tau) : -INFINITY;
#else
    double lt = tau > 0 ? log(tau) : -INFINITY;
#endif
    /* pass 1: counts per row */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < n; ++i) {
        long long c0 = 0;
        for (int j = 0; j < m; ++j) {
            double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
            double mu = -INFINITY;
            if (dirs & 1) {
                double s = (g[j] - c) / eps + log(b[j]);
#if ORC_MUTANT == 14
                double v = (tau > 0) ? s - (Mc[j] + lt) : INFINITY; /* row test against a column maximum */
#else
                double v = (tau > 0) ? s - (Mr[i] + lt) : INFINITY;
#endif
                if (v > mu) mu = v;
            }
            if (dirs & 2) {
                double s = (f[i] - c) / eps + log(a[i]);
                double v = (tau > 0) ? s - (Mc[j] + lt) : INFINITY;
                if (v > mu) mu = v;
            }
            if (mu >= -band) ++c0;
        }
        cnt[i + 1] = c0;
    }
    cnt[0] = 0;
    for (int i = 0; i < n; ++i) cnt[i + 1] += cnt[i];
    long long total = cnt[n];
    if (rows && cap >= total) {
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i) {
            long long o = cnt[i];
            for (int j = 0; j < m; ++j) {
                double c = cost_ij(X + (size_t)i * d, Y + (size_t)j * d, d);
                double mu = -INFINITY;
                if (dirs & 1) {
                    double s = (g[j] - c) / eps + log(b[j]);
#if ORC_MUTANT == 14
                    double v = (tau > 0) ? s - (Mc[j] + lt) : INFINITY;
#else
                    double v = (tau > 0) ? s - (Mr[i] + lt) : INFINITY;
#endif
                    if (v > mu) mu = v;
                }
                if (dirs & 2) {
                    double s = (f[i] - c) / eps + log(a[i]);
                    double v = (tau > 0) ? s - (Mc[j] + lt) : INFINITY;
                    if (v > mu) mu = v;
                }
                if (mu >= -band) {
                    rows[o] = i;
                    cols[o] = j;
                    if (vals) vals[o] = exp((f[i] + g[j] - c) / eps + log(a[i]) + log(b[j]));
                    if (margins) margins[o] = mu;
                    ++o;
                }
            }
        }
    }
    free(Mr); free(Mc); free(cnt);
    return total;
}

/* Gradient on a stored support: grad_i = 2 sum_{(i,j) in S} P_ij (x_i - y_j). */
/*
 * Sparse APML on a stored support (row-major COO of one cloud: rows ascending,
 * columns ascending within a row), temperature T, `iters` normalisations:
 *   s_ij   = -C_ij / T                                    on the support
 *   R_ij   = exp(s_ij) / sum_{j' in row i} exp(s_ij')      row softmax
 *   K_ij   = exp(s_ij) / sum_{i' in column j} exp(s_i'j)   column softmax
 *   P_ij   = (R_ij + K_ij) / 2                             bidirectional symmetrisation
 *   repeat iters times: P_ij *= a_i / sum_j P_ij, then P_ij *= b_j / sum_i P_ij
 *   loss   = sum P_ij C_ij
 * (empty rows and columns are left alone).  vals receives P; loss is optional.
 */
int orc_apml_coo(int n, int m, int d, const double *X, const double *Y,
                 const double *a, const double *b, long long nnz,
                 const int *rows, const int *cols, double T, int iters,
                 double *vals, double *loss) {
    if (n <= 0 || m <= 0 || d <= 0 || !(T > 0) || iters < 0 || nnz < 0) return -1;
    for (long long e = 0; e < nnz; ++e)
        if (rows[e] < 0 || rows[e] >= n || cols[e] < 0 || cols[e] >= m) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
    double *rmax = (double *)malloc(sizeof(double) * (size_t)n);
    double *rsum = (double *)malloc(sizeof(double) * (size_t)n);
    double *cmax = (double *)malloc(sizeof(double) * (size_t)m);
    double *csum = (double *)malloc(sizeof(double) * (size_t)m);
    if (!s || !rmax || !rsum || !cmax || !csum) {
        free(s); free(rmax); free(rsum); free(cmax); free(csum);
        return -2;
    }
    for (int i = 0; i < n; ++i) { rmax[i] = -INFINITY; rsum[i] = 0.0; }
    for (int j = 0; j < m; ++j) { cmax[j] = -INFINITY; csum[j] = 0.0; }
    for (long long e = 0; e < nnz; ++e) {
        s[e] = -cost_ij(X + (size_t)rows[e] * d, Y + (size_t)cols[e] * d, d) / T;
        if (s[e] > rmax[rows[e]]) rmax[rows[e]] = s[e];
        if (s[e] > cmax[cols[e]]) cmax[cols[e]] = s[e];
    }
    for (long long e = 0; e < nnz; ++e) {
        rsum[rows[e]] += exp(s[e] - rmax[rows[e]]);
        csum[cols[e]] += exp(s[e] - cmax[cols[e]]);
    }
    for (long long e = 0; e < nnz; ++e) {
        const double r = exp(s[e] - rmax[rows[e]]) / rsum[rows[e]];
        const double k = exp(s[e] - cmax[cols[e]]) / csum[cols[e]];
#if ORC_MUTANT == 11
        vals[e] = r; /* mutant: the column softmax is dropped */
        (void)k;
#else
        vals[e] = 0.5 * (r + k);
#endif
    }
    for (int it = 0; it < iters; ++it) {
        for (int i = 0; i < n; ++i) rsum[i] = 0.0;
        for (long long e = 0; e < nnz; ++e) rsum[rows[e]] += vals[e];
        for (long long e = 0; e < nnz; ++e) vals[e] *= a[rows[e]] / rsum[rows[e]];
        for (int j = 0; j < m; ++j) csum[j] = 0.0;
        for (long long e = 0; e < nnz; ++e) csum[cols[e]] += vals[e];
        for (long long e = 0; e < nnz; ++e) vals[e] *= b[cols[e]] / csum[cols[e]];
    }
    if (loss) {
        double l = 0.0;
        for (long long e = 0; e < nnz; ++e)
            l += vals[e] * cost_ij(X + (size_t)rows[e] * d, Y + (size_t)cols[e] * d, d);
        *loss = l;
    }
    free(s); free(rmax); free(rsum); free(cmax); free(csum);
    return 0;
}

int orc_grad_support(int n, int m, int d, const double *X, const double *Y,
                     long long nnz, const int *rows, const int *cols,
                     const double *vals, double *grad) {
    if (g_cost != 0) return -1; /* squared-Euclidean support gradient only */
    for (long long k = 0; k < (long long)n * d; ++k) grad[k] = 0.0;
    for (long long e = 0; e < nnz; ++e) {
        int i = rows[e], j = cols[e];
        if (i < 0 || i >= n || j < 0 || j >= m) return -1;
        for (int k = 0; k < d; ++k)
            grad[(size_t)i * d + k] += 2.0 * vals[e] * (X[(size_t)i * d + k] - Y[(size_t)j * d + k]);
    }
    return 0;
}

/*
 * Hessian-vector product of the entropic OT loss with respect to X
 * ("FlashSinkhorn", Methodologie 3, HVP paragraph: the page streams the
 * product as transport-vector and transport-matrix products and gives no
 * formula; this is the plain reading, written out densely).
 *
 * At the optimum the loss's gradient is G_i = 2 sum_j P_ij (x_i - y_j).
 * P depends on X through C and through the optimal potentials.  Moving X
 * along V (t -> X + t V) changes, to first order,
 *   C_ij  by  Cd_ij = 2 (x_i - y_j) . v_i
 *   P_ij  by  P_ij (fd_i + gd_j - Cd_ij) / eps,
 * where (fd, gd) keep both marginals of P fixed:
 *   r_i fd_i + sum_j P_ij gd_j = alpha_i := sum_j P_ij Cd_ij
 *   sum_i P_ij fd_i + c_j gd_j = beta_j  := sum_i P_ij Cd_ij
 * (r, c: the row and column sums of P).  The system is singular along
 * (fd + t, gd - t), which leaves the change of P unchanged.  Eliminating fd:
 *   S gd = beta - P^T (alpha / r),  S = diag(c) - P^T diag(1/r) P,
 * S has the constant vector as its null space; adding (mean c / m) 1 1^T
 * makes it positive definite and picks the solution with sum gd = 0
 * (Cholesky).  Then fd_i = (alpha_i - sum_j P_ij gd_j) / r_i and
 *   (H V)_i = 2 r_i v_i + (2 / eps) sum_j P_ij (fd_i + gd_j - Cd_ij) (x_i - y_j).
 * Dense: O(n m + m^2) memory and O(n m^2 + m^3) time, small problems only.
 * Squared-Euclidean cost only (returns -1 under the cosine cost).
 * fd [n] and gd [m] may be NULL.
 */
int orc_hvp(int n, int m, int d, const double *X, const double *Y,
            const double *a, const double *b, const double *f,
            const double *g, double eps, const double *V, double *out,
            double *fd_out, double *gd_out) {
    if (n <= 0 || m <= 0 || d <= 0 || !(eps > 0) || g_cost != 0) return -1;
    const size_t nm = (size_t)n * m;
    double *P = (double *)malloc(sizeof(double) * nm);
    double *Cd = (double *)malloc(sizeof(double) * nm);
    double *S = (double *)malloc(sizeof(double) * (size_t)m * m);
    double *r = (double *)calloc((size_t)n, sizeof(double));
    double *al = (double *)calloc((size_t)n, sizeof(double));
    double *fd = (double *)calloc((size_t)n, sizeof(double));
    double *c = (double *)calloc((size_t)m, sizeof(double));
    double *be = (double *)calloc((size_t)m, sizeof(double));
    double *gd = (double *)calloc((size_t)m, sizeof(double));
    int rc = 0;
    if (!P || !Cd || !S || !r || !al || !fd || !c || !be || !gd) {
        rc = -2;
        goto done;
    }
    /* the plan, the change of the cost, and their row and column sums */
    for (int i = 0; i < n; ++i) {
        const double *xi = X + (size_t)i * d, *vi = V + (size_t)i * d;
        for (int j = 0; j < m; ++j) {
            const double *yj = Y + (size_t)j * d;
            const double p = exp((f[i] + g[j] - cost_ij(xi, yj, d)) / eps + log(a[i]) + log(b[j]));
            double cd = 0.0;
            for (int k = 0; k < d; ++k) cd += 2.0 * (xi[k] - yj[k]) * vi[k];
            P[(size_t)i * m + j] = p;
            Cd[(size_t)i * m + j] = cd;
            r[i] += p;
            c[j] += p;
            al[i] += p * cd;
            be[j] += p * cd;
        }
    }
    /* Schur complement on gd, the gauge fixed by the rank-one term */
    {
        double cmean = 0.0;
        for (int j = 0; j < m; ++j) cmean += c[j];
        cmean /= m;
        const double shift = cmean / m;
        for (int j = 0; j < m; ++j)
            for (int l = 0; l <= j; ++l) {
                double s = (j == l ? c[j] : 0.0) + shift;
                for (int i = 0; i < n; ++i) s -= P[(size_t)i * m + j] * P[(size_t)i * m + l] / r[i];
                S[(size_t)j * m + l] = s;
                S[(size_t)l * m + j] = s;
            }
        for (int j = 0; j < m; ++j) {
#if ORC_MUTANT == 12
            gd[j] = 0.0; /* mutant: the column potentials are held fixed */
#else
            double s = be[j];
            for (int i = 0; i < n; ++i) s -= P[(size_t)i * m + j] * al[i] / r[i];
            gd[j] = s;
#endif
        }
#if ORC_MUTANT != 12
        /* Cholesky S = L L^T in place (lower triangle), then two triangular solves */
        for (int j = 0; j < m; ++j) {
            double s = S[(size_t)j * m + j];
            for (int k = 0; k < j; ++k) s -= S[(size_t)j * m + k] * S[(size_t)j * m + k];
            if (!(s > 0.0)) {
                rc = -3;
                goto done;
            }
            const double ljj = sqrt(s);
            S[(size_t)j * m + j] = ljj;
            for (int l = j + 1; l < m; ++l) {
                double t = S[(size_t)l * m + j];
                for (int k = 0; k < j; ++k) t -= S[(size_t)l * m + k] * S[(size_t)j * m + k];
                S[(size_t)l * m + j] = t / ljj;
            }
        }
        for (int j = 0; j < m; ++j) {
            double s = gd[j];
            for (int k = 0; k < j; ++k) s -= S[(size_t)j * m + k] * gd[k];
            gd[j] = s / S[(size_t)j * m + j];
        }
        for (int j = m - 1; j >= 0; --j) {
            double s = gd[j];
            for (int k = j + 1; k < m; ++k) s -= S[(size_t)k * m + j] * gd[k];
            gd[j] = s / S[(size_t)j * m + j];
        }
#endif
    }
    for (int i = 0; i < n; ++i) {
        double s = al[i];
        for (int j = 0; j < m; ++j) s -= P[(size_t)i * m + j] * gd[j];
        fd[i] = s / r[i];
    }
    /* assembly */
    for (int i = 0; i < n; ++i) {
        const double *xi = X + (size_t)i * d, *vi = V + (size_t)i * d;
        double *oi = out + (size_t)i * d;
        for (int k = 0; k < d; ++k) oi[k] = 2.0 * r[i] * vi[k];
        for (int j = 0; j < m; ++j) {
            const double *yj = Y + (size_t)j * d;
            const double w = 2.0 / eps * P[(size_t)i * m + j] * (fd[i] + gd[j] - Cd[(size_t)i * m + j]);
            for (int k = 0; k < d; ++k) oi[k] += w * (xi[k] - yj[k]);
        }
    }
    if (fd_out) memcpy(fd_out, fd, sizeof(double) * (size_t)n);
    if (gd_out) memcpy(gd_out, gd, sizeof(double) * (size_t)m);
done:
    free(P); free(Cd); free(S); free(r); free(al); free(fd); free(c); free(be); free(gd);
    return rc;
}
