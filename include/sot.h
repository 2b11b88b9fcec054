/*
 * sot.h -- C ABI of the GB300 (sm_103a) log-domain Sinkhorn library for point
 * clouds with squared-Euclidean cost.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All array pointers are DEVICE pointers (cudaMalloc'd or torch-allocated
 *   memory on the current device) unless the parameter name ends in _host.
 *   The caller owns every array; the library never allocates an output.
 * - Layout: float32, row-major, contiguous, batch-major:
 *     X[B][n][d], Y[B][m][d]          point clouds (source rows, target columns)
 *     a[B][n], b[B][m]                probability weights; NULL = uniform 1/n, 1/m
 *     f[B][n], g[B][m]                dual potentials (true, unshifted values)
 *   Weights must be > 0 and finite, each a[k] and b[k] summing to one.
 * - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call is stream-ordered.  Calls are asynchronous unless documented
 *   otherwise; scratch memory is taken stream-ordered on `stream` and released
 *   before the call returns its status.  It comes from a pool per device that
 *   the library creates on first use and keeps for the life of the process;
 *   the pool holds up to 2 GiB of released scratch for later calls and
 *   returns the rest to the driver.
 * - Every call returns an int status (SOT_OK = 0 or a negative SOT_ERR_*)
 *   and never throws or aborts.  Arguments are checked on the host before
 *   anything is launched; on error, output contents are unspecified except
 *   where stated.  sot_last_error() gives a one-line description of the most
 *   recent failure on the calling thread.
 * - Non-finite inputs are not detected by the asynchronous calls (they
 *   propagate into the outputs); sot_check_inputs() validates synchronously.
 *
 * Notation (page "FlashSinkhorn: IO-aware entropic optimal transport on GPU",
 * Methodologie 1, Propositie 1):
 *   C_ij = |x_i - y_j|^2,  P_ij = a_i b_j exp((f_i + g_j - C_ij) / eps)
 *   f-half:  f_i <- -eps LSE_j[(g_j - C_ij)/eps + log b_j]
 *   g-half:  g_j <- -eps LSE_i[(f_i - C_ij)/eps + log a_i]
 * One iteration is an f-half followed by a g-half that uses the new f.  The
 * kernels evaluate each half as a row-wise LSE of the biased dot-product
 * score (2 x_i.y_j + g_j - |y_j|^2 + eps log b_j)/eps, streaming tiles of the
 * other cloud; the n x m cost matrix is never stored (same page,
 * Methodologie 2).
 */
#ifndef SOT_H
#define SOT_H

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum sot_status {
    SOT_OK = 0,
    SOT_ERR_INVALID_ARG = -1,  /* bad size, NULL pointer, eps <= 0, ... */
    SOT_ERR_NONFINITE = -2,    /* sot_check_inputs: NaN/Inf coordinate or weight, or weight <= 0 */
    SOT_ERR_CAPACITY = -3,     /* sot_plan_coo: capacity < nnz; *nnz_host holds the required count */
    SOT_ERR_TIMEOUT = -4,      /* a bounded device-side wait gave up */
    SOT_ERR_CUDA = -5,         /* a CUDA runtime call or launch failed */
    SOT_ERR_UNSUPPORTED = -6,  /* the requested precision / size has no kernel on this device */
    SOT_ERR_NOMEM = -7         /* stream-ordered scratch allocation failed */
};

/* ---- schedule flags ---------------------------------------------------- */
enum sot_flags {
    SOT_PREC_AUTO = 0,          /* d <= 3: point path (fp32 FMA); 4 <= d <= 16: fp32 FMA; 17 <= d <= 1024: tensor
                                   cores (fp16 x3) at d = 64, 128, 192, 256, 512 or 1024, other d zero-padded to
                                   the next of these */
    SOT_PREC_FP32 = 1,          /* fp32 FMA contraction for any d <= 1024 (above 256 the coordinates stream in
                                   slices of 256) */
    SOT_PREC_F16X3 = 2,         /* tcgen05 fp16 products hi*hi + hi*lo + lo*hi (fp32-class accuracy), any
                                   4 <= d <= 1024 (zero-padded as above) */
    SOT_PREC_MASK = 3,
    SOT_WARM_START = 1 << 4,    /* read f, g as the initial potentials instead of f = g = 0 */
    SOT_STAGE_EARLY_EXIT = 1 << 5, /* apply the stop test in every stage, not only at the final eps */
    SOT_TC_NO_SCREEN = 1 << 6,     /* tensor path: evaluate every pair's exponential in every half-step
                                      (default: warm half-steps screen pairs with hi*hi products first) */
    SOT_NO_CLUSTER = 1 << 7,       /* point path: stream every half-step (default: when both clouds fit in
                                      shared memory, the warm iterations of an untested stage run in one
                                      cluster-resident launch) */
    SOT_COST_COSINE = 1 << 8       /* cosine cost C_ij = 2 - 2 x_i.y_j / (|x_i| |y_j|) ("FlashSinkhorn",
                                      Conclusies: the cost structure holds for the cosine distance after
                                      normalisation).  Every step runs on the unit points x/|x|, y/|y|, where
                                      |xhat - yhat|^2 equals that cost; a zero point stays the zero vector (its
                                      cost to a unit point is 1, gradient 0).  Plan application carries the
                                      gradient back through x/|x|.  Accepted by sot_potentials_ex and
                                      sot_plan_apply; the potentials and plan are those of the cosine cost. */
};

/*
 * Annealing schedule.  Stages k = 0, 1, ... use eps_k = max(eps, eps_init * eps_factor^k);
 * the first k with eps_init * eps_factor^k <= eps is the last stage (clamped
 * to eps).  eps_init <= eps (or eps_factor outside (0,1)) means one stage at eps.
 * Every stage runs iters_per_stage iterations, warm-started from the previous one.
 * Stop test (tol > 0): after an iteration at the final eps (or in any stage
 * with SOT_STAGE_EARLY_EXIT) the row-marginal error sum_i |sum_j P_ij - a_i|
 * of the current (f, g) is compared with tol, using the largest error over the
 * batch; passing ends the stage (the solve, at the final eps).  The final
 * stage continues past iters_per_stage until the test passes or the total
 * number of iterations reaches max_iters (max_iters <= 0: no extension).
 * eps annealing and the stop rule are not fixed by the pages; this is the
 * reading this library implements.
 */
typedef struct {
    float eps;            /* final (or only) eps, > 0 */
    float eps_init;       /* first-stage eps (annealing when > eps) */
    float eps_factor;     /* per-stage factor in (0, 1) */
    int iters_per_stage;  /* >= 0 */
    int max_iters;        /* cap on total iterations (<= 0: stages only) */
    float tol;            /* stop tolerance on the marginal error (<= 0: none) */
    int flags;            /* sot_flags */
} sot_schedule;

/* Filled by sot_potentials_ex when non-NULL (the call then synchronises `stream`). */
typedef struct {
    int iters_done;        /* total iterations returned */
    int stages_done;       /* stages entered */
    int converged;         /* 1 if the stop test passed at the final eps */
    float final_eps;
    float* err_host;       /* [B] or NULL: marginal error of the returned iterate (NaN if not evaluated) */
    int* stage_iters_host; /* [stage_iters_cap] or NULL: iterations realised per stage */
    int stage_iters_cap;
} sot_stats;

/* ---- calls --------------------------------------------------------------- */

/*
 * Fixed schedule: `iters` iterations at `eps` from f = g = 0.  Asynchronous.
 * Page: "FlashSinkhorn", Methodologie 1 (the update) and 2 (fused streaming).
 */
int sot_potentials(const float* X, const float* Y, const float* a, const float* b,
                   int B, int n, int m, int d, float eps, int iters,
                   float* f, float* g, void* stream);

/*
 * General schedule (annealing, stop test, warm start, precision), see
 * sot_schedule.  Synchronises `stream` when st != NULL, or when the stop test
 * is active (it reads a device flag every few iterations).  The tensor-core
 * half-steps bound every device-side wait (2 s); one that gives up leaves NaN
 * potentials, and a call with st != NULL then returns SOT_ERR_TIMEOUT (a call
 * without st reports it through sot_async_status).
 */
int sot_potentials_ex(const float* X, const float* Y, const float* a, const float* b,
                      int B, int n, int m, int d, const sot_schedule* s,
                      float* f, float* g, sot_stats* st, void* stream);

/*
 * Plan application with the given (f, g) at eps, without storing P
 * ("FlashSinkhorn", Methodologie 3):
 *   cost[k]     = sum_ij P_ij C_ij                        (may be NULL)
 *   grad[k][i]  = 2 (a_i x_i - sum_j P_ij y_j)  [B][n][d] (may be NULL)
 *   rowsum[k][i]= sum_j P_ij                    [B][n]    (may be NULL)
 * Asynchronous.  flags: SOT_PREC_* (0 = auto), optionally | SOT_COST_COSINE (the
 * potentials must then be those of the cosine cost; the gradient is carried back
 * through x/|x|).
 */
int sot_plan_apply(const float* X, const float* Y, const float* a, const float* b,
                   int B, int n, int m, int d, const float* f, const float* g, float eps,
                   float* cost, float* grad, float* rowsum, int flags, void* stream);

/*
 * Transport-matrix products with the given (f, g) at eps, streamed without
 * storing P ("FlashSinkhorn", Methodologie 3 and its HVP paragraph: the
 * Hessian-vector product decomposes into transport-vector and
 * transport-matrix products), P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps):
 *   side 0: out[k][i][:] = sum_j P_ij V[k][j][:]    V [B][m][c] -> out [B][n][c]
 *   side 1: out[k][j][:] = sum_i P_ij V[k][i][:]    V [B][n][c] -> out [B][m][c]
 * c = 1 is a transport-vector product; 1 <= c <= 64, d <= 256.  Pairs whose
 * weight is below 2^-30 / (number of summed points) of a_i (side 0) or b_j
 * (side 1) are skipped, under 2^-30 of it in all; every
 * other pair's P_ij is evaluated in float-float arithmetic from the caller's
 * coordinates and potentials.  flags: 0 or SOT_COST_COSINE.  V and out are
 * device arrays owned by the caller; out is fully written.  Asynchronous.
 */
int sot_transport_apply(const float* X, const float* Y, const float* a, const float* b,
                        int B, int n, int m, int d, const float* f, const float* g, float eps,
                        const float* V, int c, int side, float* out, int flags, void* stream);

/*
 * Gradient with respect to Y with the given (f, g) at eps, the mirror of the
 * gradient of sot_plan_apply: grad_y[k][j] = 2 (b_j y_j - sum_i P_ij x_i),
 * [B][m][d], formed from the transport product P^T X (see
 * sot_transport_apply; d <= 256).  flags: 0 or SOT_COST_COSINE (then the
 * gradient is carried back through y/|y|).  Asynchronous.
 */
int sot_grad_y(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
               const float* f, const float* g, float eps, float* grad_y, int flags, void* stream);

/*
 * Hessian-vector product of the entropic OT loss with respect to X
 * ("FlashSinkhorn", Methodologie 3, HVP paragraph: streamed as transport-vector
 * and transport-matrix products, P never stored).  Reading: the Hessian of the
 * converged loss, whose gradient is 2 sum_j P_ij (x_i - y_j), with the
 * potentials' first-order change keeping both marginals fixed:
 *   out = H V,  V and out [B][n][d] fp32 device arrays (row-major, caller-owned).
 * The marginal system is solved by conjugate gradients preconditioned with the
 * column sums of P: at most cg_iters steps, all clouds at once, stopping when
 * every cloud's preconditioned residual has fallen to cg_tol of its start
 * (checked every 8 steps; a cloud that is done keeps its solution).  Each step
 * is one P u and one P^T u.  The assembly forms its sums pair by pair around
 * each row's barycentre.  The clouds are first moved by their common centre
 * (H does not change).  Squared-Euclidean cost, d <= 9, flags must be 0.  f, g
 * are the potentials the plan is built from (converged ones for the Hessian of
 * the loss).  Synchronises `stream` every 8 CG steps; scratch O((n + m) d).
 * Errors: SOT_ERR_INVALID_ARG (sizes, eps, cg arguments, NULL pointers, flags),
 * SOT_ERR_UNSUPPORTED (d > 9), SOT_ERR_NOMEM, SOT_ERR_CUDA.
 */
int sot_hvp(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
            const float* f, const float* g, float eps, const float* V, int cg_iters, float cg_tol, float* out,
            int flags, void* stream);

/* Convenience forms of sot_plan_apply (precision auto). */
int sot_cost(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
             const float* f, const float* g, float eps, float* cost, void* stream);
int sot_grad_x(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
               const float* f, const float* g, float eps, float* grad, void* stream);
int sot_cost_grad(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                  const float* f, const float* g, float eps, float* cost, float* grad, void* stream);

/*
 * Thresholded COO plan ("From Theory to Throughput: CUDA-Optimized APML",
 * Abstract and Innovation: thresholded assignments, bidirectional
 * symmetrisation, COO storage).  With s_ij = (g_j - C_ij)/eps + log b_j and
 * s'_ij = (f_i - C_ij)/eps + log a_i, pair (i, j) is kept when
 *   (dirs & 1) and s_ij  >= max_j' s_ij'  + log(threshold)   [P_ij >= threshold * row max], or
 *   (dirs & 2) and s'_ij >= max_i' s'_i'j + log(threshold)   [P_ij >= threshold * column max].
 * threshold in [0, 1]; 0 keeps every pair.  Output, cloud after cloud, row-major
 * (row ascending, then column ascending) with cloud-local int32 indices:
 *   rows[nnz], cols[nnz], vals[nnz] = P_ij (fp32), batch_offsets[B+1] (int64, device).
 * Synchronises `stream` once (to read the count).  *nnz_host (host) always
 * receives the total count; if it exceeds capacity the call returns
 * SOT_ERR_CAPACITY and writes no entries.
 */
int sot_plan_coo(const float* X, const float* Y, const float* a, const float* b,
                 int B, int n, int m, int d, const float* f, const float* g, float eps,
                 float threshold, int dirs, long long capacity,
                 int* rows, int* cols, float* vals, long long* batch_offsets,
                 long long* nnz_host, void* stream);

/*
 * The fp32 operands that sot_plan_coo's predicate reads, for auditing its
 * decisions ("CUDA-Optimized APML", Abstract / Innovation: the thresholded
 * support).  Given the same inputs as sot_plan_coo, it writes (device arrays
 * owned by the caller):
 *   xc[B][n][d], yc[B][m][d]  coordinates less the common per-cloud shift
 *                             t = (mean x + mean y) / 2 (the cost is unchanged);
 *   lwx[B][n], lwy[B][m]      log2 of the weights (log2(1/n) when a is NULL);
 *   Lx[B][n], Ly[B][m]        the base-2 states of f and g, kappa = 1 / (eps ln 2):
 *                             Lx = kappa (|xc|^2 - f) for d > 3 and kappa (0 - f) for d <= 3;
 *   Mr[B][n], Mc[B][m]        the row and column maxima of the two scores;
 * and scalars_host[2] = { kappa, log2(threshold) } (host).  Every kept or
 * dropped pair of sot_plan_coo is decided from these values alone, with
 * single rounding (round to nearest even) at every step, by:
 *   d <= 3 (k ascending, u = fl(sqrt(kappa) xc), v = fl(sqrt(kappa) yc)):
 *     row score  t_ij = -fma chain over k of (fl(u_ik - v_jk))^2 started at -fl(lwy_j - Ly_j);
 *     col score  t'_ij = -fma chain over k of (fl(v_jk - u_ik))^2 started at -fl(lwx_i - Lx_i);
 *   d > 3: p_ij = fma chain over k of xc_ik yc_jk from 0;
 *     t_ij = fma(2 kappa, p_ij, fl(lwy_j - Ly_j)), t'_ij = fma(2 kappa, p_ij, fl(lwx_i - Lx_i));
 *   Mr_i = max_j t_ij, Mc_j = max_i t'_ij, and pair (i, j) is kept when
 *   (dirs & 1) and t_ij >= fl(Mr_i + log2 tau), or (dirs & 2) and t'_ij >= fl(Mc_j + log2 tau).
 * Asynchronous on `stream`; same argument errors as sot_plan_coo.
 */
int sot_plan_coo_operands(const float* X, const float* Y, const float* a, const float* b,
                          int B, int n, int m, int d, const float* f, const float* g, float eps,
                          float threshold, float* xc, float* lwx, float* Lx, float* yc, float* lwy,
                          float* Ly, float* Mr, float* Mc, float* scalars_host, void* stream);

/*
 * Sparse APML on a stored support ("From Theory to Throughput: CUDA-Optimized
 * APML", Abstract and Innovation: an adaptive softmax, bidirectional
 * symmetrisation and Sinkhorn normalisation run directly in COO form, and
 * gradients are kept on the stored support).  The support is a row-major COO
 * such as sot_plan_coo returns (rows ascending within a cloud, cloud-local
 * int32 indices, int64 batch_offsets[B+1] from 0 to nnz; device arrays).
 * With s_ij = -C_ij / T on the stored pairs:
 *   P = (row softmax of s + column softmax of s) / 2, then `iters` times the
 *   rows are scaled to sum to a_i and the columns to sum to b_j;
 *   vals[nnz]  <- P on the support (fp32);
 *   loss[B]    <- sum P_ij C_ij (may be NULL);
 *   grad[B][n][d] <- 2 sum_j P_ij (x_i - y_j) on the support, P held fixed (may be NULL).
 * T > 0 is the temperature (the page's adaptive temperature is not given; a
 * caller passes one, e.g. eps).  The offsets and the support are checked on the
 * device before any entry is read through them: offsets that do not run
 * non-decreasing from 0 to nnz, unsorted rows or an out-of-range index return
 * SOT_ERR_INVALID_ARG.  Synchronises the stream once, at the end, to read that
 * check (twice with a gradient at d > 3).  nnz < 2^31.
 */
int sot_apml_coo(const float* X, const float* Y, const float* a, const float* b,
                 int B, int n, int m, int d, const int* rows, const int* cols,
                 const long long* batch_offsets, long long nnz, float T, int iters,
                 float* vals, float* loss, float* grad, void* stream);

/*
 * Gradient on a stored support ("CUDA-Optimized APML", Innovation: gradients
 * preserved on the stored support):
 *   grad[k][i] = 2 sum_{e in cloud k, rows[e] = i} vals[e] (x_i - y_cols[e])
 * The COO must be row-sorted within each cloud (as sot_plan_coo writes it);
 * unsorted or out-of-range entries make the call return SOT_ERR_INVALID_ARG
 * (checked on the device).  batch_offsets is a device array [B+1] whose last
 * element is the number of entries.  The call synchronises `stream` once to
 * read the check's result.
 */
int sot_grad_x_coo(const float* X, const float* Y, int B, int n, int m, int d,
                   const int* rows, const int* cols, const float* vals,
                   const long long* batch_offsets, float* grad, void* stream);

/*
 * Synchronous input validation: every coordinate finite, every weight finite
 * and > 0.  Returns SOT_OK, SOT_ERR_NONFINITE or SOT_ERR_INVALID_ARG.
 */
int sot_check_inputs(const float* X, const float* Y, const float* a, const float* b,
                     int B, int n, int m, int d, void* stream);

/*
 * Per-kernel timing with CUDA events recorded on the launching stream around
 * every half-step launch (off by default).  sot_profile_read synchronises the
 * device events, returns the number of half-steps since the last reset (a
 * cluster-resident launch counts the half-steps it covers) and their summed
 * duration in milliseconds, and resets the counters.
 */
int sot_profile_enable(int on);
int sot_profile_read(long long* launches_host, double* total_ms_host);
/*
 * The same, split by kind: index 0 counts streaming half-steps that form
 * every pair's exponential, index 1 the screened tensor-core half-steps,
 * index 2 the half-steps run inside cluster-resident launches (one launch
 * covers many; its time is counted once).  Counts are half-steps, times are
 * milliseconds.  Both arrays (host, 3 entries each) may be NULL.  Resets the
 * counters like sot_profile_read.
 */
int sot_profile_read_kinds(long long* launches_host, double* ms_host);

/*
 * sot_potentials without any memory allocation.  No counterpart in the source
 * pages: this entry serves callers that cannot allocate device memory on the
 * call path -- for example a process whose device memory is entirely reserved
 * up front by another framework's caching allocator, or real-time and
 * latency-critical loops where an allocator call (and the synchronisation or
 * pool growth it can trigger) is not allowed.
 *
 * Same computation and result as sot_potentials (fixed schedule, f = g = 0
 * start) for point clouds with d <= 3.  Its scratch is one statically sized
 * device array of SOT_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the
 * library until the process exits; a problem whose scratch would not fit is
 * rejected with SOT_ERR_INVALID_ARG (sot_last_error() gives the bytes it would
 * need) before anything runs, and d > 3 gives SOT_ERR_UNSUPPORTED.  The call
 * makes no cudaMalloc / cudaFree / cudaMallocAsync / cudaMallocFromPoolAsync call.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call reuses the same array and clears what
 * must start at zero, so calls that overlap on the GPU (other streams, other
 * host threads on the same device) race on it: serialise them.
 */
#define SOT_NOALLOC_SCRATCH_BYTES (16u << 20)
int sot_potentials_noalloc(const float* X, const float* Y, const float* a, const float* b,
                           int B, int n, int m, int d, float eps, int iters,
                           float* f, float* g, void* stream);

/*
 * Device-side status of the asynchronous calls (sot_potentials,
 * sot_potentials_ex without stats, sot_plan_apply and its convenience forms)
 * made on the current device since the last sot_async_status.  Synchronises
 * `stream` (give the stream of those calls, or NULL after synchronising them),
 * returns SOT_ERR_TIMEOUT when a bounded device-side wait of a tensor-core
 * kernel gave up in one of them (the rows that kernel held are NaN) and
 * SOT_OK otherwise, and clears the status.
 */
int sot_async_status(void* stream);

/*
 * Testing hook for the timeout path of the tensor-core kernels.  With
 * tile >= 0, the tensor-core kernels launched after the next
 * `after_launches` ones issue no bulk copy from column tile `tile` of their
 * column chunk onward, so their waits on that tile run out after wait_ns
 * nanoseconds (wait_ns <= 0: the default 2 s): such a kernel waits for the
 * copies and MMAs it did issue, frees TMEM, leaves NaN rows and reports
 * SOT_ERR_TIMEOUT as above.  tile < 0 turns the hook off and restores the
 * default limit.  Process-wide and not synchronised with work in flight: set
 * it between calls.  Not for production use.
 */
int sot_test_hold_tile(int tile, int after_launches, long long wait_ns);

/*
 * Which kernel family a solve of dimension d with these flags would use:
 * 0 = fp32 point kernels (d <= 3), 1 = fp32 dense kernels, 2 = tcgen05
 * tensor-core kernels; or a negative SOT_ERR_* when none applies.  Host only.
 */
int sot_select_path(int d, int flags);

/* Number of CUDA kernels this library has launched since it was loaded
 * (all devices, all threads).  Diagnostic; no synchronisation. */
long long sot_kernel_launches(void);

/* Static strings; never NULL. */
const char* sot_status_string(int status);
const char* sot_last_error(void);
int sot_version(void); /* major * 10000 + minor * 100 + patch */

#ifdef __cplusplus
}
#endif
#endif /* SOT_H */
