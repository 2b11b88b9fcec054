// kernels.h -- launcher interface between the C ABI (sot_api.cu) and the
// kernel sources.  Internal to libsot; not installed.
//
// Internal state of a solve (all device arrays, batch-major):
//   point path (d <= 3): xpack[B][n], ypack[B][m] are float4 (x - t, log2 a)
//     with t the per-cloud centring translation (C is translation invariant)
//     and unused coordinates zero;
//   dense / tensor paths: xc[B][n][d], yc[B][m][d] centred coordinates plus
//     log2 weights lw2x[B][n], lw2y[B][m];
//   nx[B][n], ny[B][m]: squared norms of the centred points (dense and tensor
//     paths); zero for the point path;
//   L[B][n], Lam[B][m]: row / column log2-LSE values.  With kappa = 1/(eps ln 2),
//     f_i = nx_i - L_i / kappa and g_j = ny_j - Lam_j / kappa.
// Dense / tensor f-half (expanded form):
//     L_i = log2 sum_j 2^(2 kappa x_i.y_j + lw2y_j - Lam_j)
// Point f-half (direct form, nx = ny = 0, so L_i = -kappa f_i):
//     L_i = log2 sum_j 2^(lw2y_j - Lam_j - kappa |x_i - y_j|^2)
// The g-halves are the mirror images.
#pragma once
#include <cuda_runtime.h>

namespace sot {

// Number of kernels this library has launched (every launcher adds its own).
void count_launches(int k);
long long launches_total();

enum HalfMode { MODE_LSE = 0, MODE_MAX = 1 };

struct HalfArgs {
    int B, nr, nc, d;
    const float* rpack;     // point: float4 [B][nr]; dense: [B][nr][d] centred rows
    const float* cpack;     // point: float4 [B][nc]; dense: [B][nc][d] centred columns
    const float* cw2;       // dense: column log2 weights [B][nc] (point: in cpack .w)
    const float* cstate;    // column state [B][nc]; column bias c_j = w2_j - cstate_j
    const float* rstate_in; // [B][nr] previous row value (stabiliser / error reference)
    float* rstate_out;      // [B][nr] (may alias rstate_in)
    const float* rweight;   // [B][nr] linear row weights for the error (NULL = uniform)
    float two_kappa;        // 2 / (eps ln 2)
    int cold;               // 1: no previous row value (stabiliser starts at -inf)
    int split, chunk;       // columns split into `split` chunks of `chunk` columns
    int rowtiles;           // row tiles per cloud
    float* part_m;          // [split][B*nr] partial (m, s) when split > 1
    float* part_s;
    unsigned* counters;     // [B*rowtiles], zero between launches
    float* errpart;         // [B*rowtiles] row-marginal error partials or NULL
    const int* stop_flag;   // NULL or device flag: nonzero => kernel returns at once
    int* status;            // device status word (SOT_DEV_* bits)
    const unsigned* lo_in;  // [B] stabiliser bound from the other side (ord-encoded) or NULL
    unsigned* lo_out;       // [B] receives min over rows of (old - new) (ord-encoded) or NULL
    unsigned* lo_reset;     // [B] slot reset to SOT_ORD_EMPTY by block (0,0) or NULL
    int* redo;              // NULL, or [B*rowtiles] row-block flags: the screened half-step sets the flag of
                            // a row block it leaves to the full half-step; the full half-step then runs
                            // only the flagged row blocks
    int rpt = 4;            // point path: rows per thread (point_plan); rowtiles = ceil(nr / (128 rpt))
};

struct ApplyArgs {
    int B, n, m, d;
    const float* xpack;   // point: float4; dense: centred [B][n][d]
    const float* ypack;
    const float* lw2x;    // dense only
    const float* lw2y;
    const float* nx;
    const float* ny;
    const float* L;
    const float* Lam;
    const float* X;       // original coordinates (gradient)
    const float* a;       // linear weights or NULL (uniform)
    const float* shift;   // [B][d] centring translation
    float kappa;          // 1 / (eps ln 2)
    int rowtiles;
    float* cost_part;     // [B*rowtiles] or NULL
    float* grad;          // [B][n][d] or NULL
    float* rowsum;        // [B][n] or NULL
    const float* Yorig;   // original target coordinates (exact pair terms)
    const float* fpot;    // caller's potentials (exact pair terms)
    const float* gpot;
    double kappa64;       // 1 / (eps ln 2) in double
    int exact_sig = 0;    // dense path: re-evaluate each significant pair's weight exactly (float-float)
};

struct CooArgs {
    int B, n, m, d;
    const float* xpack, *ypack, *lw2x, *lw2y, *nx, *ny, *L, *Lam;
    const float* Mr;      // [B][n] row maxima of the f-side score (log2)
    const float* Mc;      // [B][m] column maxima of the g-side score (log2)
    const float* a;       // linear weights or NULL
    const float *X, *Y;   // the caller's points [B][n][d], [B][m][d] (stored values)
    const float *f, *g;   // the caller's potentials (stored values)
    float two_kappa, kappa, log2tau;
    float kap_hi, kap_lo; // 1 / (eps ln 2) as a float-float pair (stored values)
    int dirs;
    int* counts;               // [B*n] count pass output
    const long long* rowptr;   // [B*n+1] write pass input (global offsets)
    long long capacity;        // entries the output arrays hold (writes at or past it are dropped)
    int* rows;
    int* cols;
    float* vals;
};

// ---- point path (d <= 3), k_point.cu ----
int point_cols_per_tile();
// Rows per thread (1, 2 or 4), column split and row tiles of a half-step over
// B clouds of nr rows and nc columns (the plan of least estimated time).
void point_plan(int B, int nr, int nc, int sms, int* rpt, int* split, int* chunk, int* rowtiles);
cudaError_t launch_point_half(const HalfArgs& p, int mode, cudaStream_t st);
int point_apply_rows_per_cta();
cudaError_t launch_point_apply(const ApplyArgs& p, cudaStream_t st);
cudaError_t launch_point_coo(const CooArgs& p, int write_pass, cudaStream_t st);

// ---- cluster-resident iterations for small point clouds, k_cluster.cu ----
size_t cluster_smem_bytes(int n, int m);
bool point_cluster_plan(int B, int n, int m, int sms, int* C, int* T, int* S, size_t* smem);
// `iters` warm iterations (f-half, then g-half) on the states L, Lam in place;
// cudaErrorInvalidConfiguration when no cluster of this shape fits the device.
cudaError_t launch_point_cluster(int B, int n, int m, const float* xpack, const float* ypack, float* L, float* Lam,
                                 float two_kappa, int iters, int C, int T, int S, size_t smem, cudaStream_t st);

// ---- dense fp32 path (any d <= 1024), k_dense.cu ----
int dense_rows_per_cta();
int dense_cols_per_tile();
int dense_max_d();
cudaError_t launch_dense_half(const HalfArgs& p, int mode, cudaStream_t st);
int dense_apply_rows_per_cta();
cudaError_t launch_dense_apply(const ApplyArgs& p, cudaStream_t st);
cudaError_t launch_dense_coo(const CooArgs& p, int write_pass, cudaStream_t st);

// ---- preprocessing and small kernels, k_prep.cu ----
// Cosine cost: unit directions of `count` points, and the gradient carried
// back through x / |x| (in place).
cudaError_t launch_normalise(const float* P, long long count, int d, float* out, cudaStream_t st);
cudaError_t launch_pad(const float* src, long long count, int d, int D, float* dst, cudaStream_t st);
cudaError_t launch_cosine_grad(const float* X, long long count, int d, float* grad, cudaStream_t st);
cudaError_t launch_center(const float* X, const float* Y, int B, int n, int m, int d,
                          float* shift, cudaStream_t st);
cudaError_t launch_pack(const float* P, const float* w, int B, int n, int d, const float* shift,
                        int point_layout, float* pack, float* lw2, float* nrm, cudaStream_t st);
cudaError_t launch_state_from_potential(const float* nrm, const float* pot, float kappa, int count,
                                        float* state, cudaStream_t st);
cudaError_t launch_potential_from_state(const float* nrm, const float* state, float kappa, int count,
                                        float* pot, cudaStream_t st);
cudaError_t launch_state_cold(const float* nrm, float kappa, int count, float* state, cudaStream_t st);
cudaError_t launch_scale(float* v, float s, int count, cudaStream_t st);
cudaError_t launch_copy(float* dst, const float* src, int count, const int* stop_flag, cudaStream_t st);
cudaError_t launch_reduce_parts(const float* part, int B, int parts, float* out, cudaStream_t st);
// Stop test: err[b] = sum of errpart[b][*]; passes when max_b err[b] < tol.
// On pass (or when force_stop) sets *stop_flag; otherwise copies L_next -> L_cur.
cudaError_t launch_decide(const float* errpart, int B, int parts, float tol, int force_stop,
                          float* err_out, int* stop_flag, int* conv_flag, const float* L_next,
                          float* L_cur, int count, cudaStream_t st);
cudaError_t launch_count_iter(const int* stop_flag, int* counter, cudaStream_t st);
// OR a call's status word into the device's word for asynchronous calls.
cudaError_t launch_status_merge(const int* status, cudaStream_t st);
// Read and clear that word (synchronises `st`).
cudaError_t read_clear_async_status(cudaStream_t st, unsigned* out);
cudaError_t launch_check_inputs(const float* X, const float* w, long long count_pts, int d,
                                long long count_w, int* bad, cudaStream_t st);
cudaError_t launch_scan_counts(const int* counts, int B, int n, long long* rowptr,
                               long long* batch_offsets, cudaStream_t st);
cudaError_t launch_grad_coo(const float* X, const float* Y, int B, int n, int m, int d,
                            const int* rows, const int* cols, const float* vals,
                            const long long* batch_offsets, float* grad, int* status,
                            cudaStream_t st);

}  // namespace sot
