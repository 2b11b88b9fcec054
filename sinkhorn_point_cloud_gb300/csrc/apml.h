// apml.h -- sparse APML on a stored COO support ("From Theory to Throughput:
// CUDA-Optimized APML", Abstract and Innovation: adaptive softmax,
// bidirectional symmetrisation and Sinkhorn normalisation run directly in COO
// form; gradients kept on the stored support).
#pragma once
#include <cuda_runtime.h>

namespace sot {

struct ApmlArgs {
    int B, n, m, d;
    const float* X;            // [B][n][d]
    const float* Y;            // [B][m][d]
    const float* a;            // [B][n] or NULL (uniform)
    const float* b;            // [B][m] or NULL (uniform)
    const int* rows;           // [nnz] cloud-local, ascending within a cloud
    const int* cols;           // [nnz] cloud-local
    const long long* off;      // [B+1] entries of cloud k: off[k] .. off[k+1]
    float inv_T;               // 1 / temperature
    int iters;                 // normalisations (row, then column)
    float* vals;               // [nnz] out: the plan on the support
    float* loss;               // [B] out or NULL
    // scratch
    float* cost;               // [nnz] C of every stored pair
    int* rstart;               // [B][n] first entry of each row (zero on entry)
    int* rend;                 // [B][n] one past its last entry (zero on entry)
    unsigned* cmax;            // [B][m] ord-encoded column maxima of s (zero on entry)
    double* csum;              // [B][m] column sums
    float* cfac;               // [B][m] per-column factor (1 / sum, or b_j / sum)
    float* loss_part;          // [B][n] per-row loss terms
    int* status;               // SOT_DEV_BAD_COO on an invalid support
};

cudaError_t launch_apml(const ApmlArgs& p, cudaStream_t st);

}  // namespace sot
