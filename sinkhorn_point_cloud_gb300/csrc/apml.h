// apml.h -- sparse APML on a stored COO support ("From Theory to Throughput:
// CUDA-Optimized APML", Abstract and Innovation: adaptive softmax,
// bidirectional symmetrisation and Sinkhorn normalisation run directly in COO
// form; gradients kept on the stored support).
#pragma once
#include <cuda_runtime.h>
#include <cstddef>

namespace sot {

struct ApmlArgs {
    int B, n, m, d;
    const float* X;            // [B][n][d]
    const float* Y;            // [B][m][d]
    const float* a;            // [B][n] or NULL (uniform)
    const float* b;            // [B][m] or NULL (uniform)
    const int* rows;           // [nnz] cloud-local, ascending within a cloud
    const int* cols;           // [nnz] cloud-local
    const long long* off;      // [B+1] entries of cloud k: off[k] .. off[k+1] (checked on the device)
    long long nnz;             // entries in all (< 2^31)
    float inv_T;               // 1 / temperature
    int iters;                 // normalisations (row, then column)
    float* vals;               // [nnz] out: the plan on the support
    float* loss;               // [B] out or NULL
    float* grad;               // [B][n][d] out or NULL: 2 sum_j P_ij (x_i - y_j), d <= 3 only
    // partition of the row passes (apml_plan)
    int cpc;                   // CTAs per cloud
    int rpc;                   // rows per CTA
    // scratch
    float* cost;               // [nnz] C of every stored pair
    int* rstart;               // [B][n] first entry of each row (zero on entry)
    int* rend;                 // [B][n] one past its last entry (zero on entry)
    float2* rstat;             // [B][n] row maximum of s and sum of exp(s - maximum)
    float* ufac;               // [B][n] row factors U
    float* cm;                 // [B][m] column maxima of s
    float* cfac;               // [B][m] 1 / column sums of exp(s - column maximum)
    float* vfac;               // [B][m] column factors V
    float* part;               // [B][cpc][m] per-CTA column partials (staged form), else NULL
    unsigned* cmax;            // [B][m] ord-encoded column maxima (global form; zero on entry)
    double* csum;              // [B][m] column sums (global form; zero on entry)
    float* loss_part;          // [B][n] per-row loss terms
    int* status;               // SOT_DEV_BAD_COO on an invalid support
};

// Row-pass partition for B clouds of n rows on `sms` SMs: fills *cpc, *rpc and
// returns the floats of per-CTA column partials the passes need (0 when the
// columns are too many to stage in shared memory: the passes then add into
// cmax / csum with global atomics).
size_t apml_plan(int B, int n, int m, int sms, int* cpc, int* rpc);
cudaError_t launch_apml(const ApmlArgs& p, cudaStream_t st);

}  // namespace sot
