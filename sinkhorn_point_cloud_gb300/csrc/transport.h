// transport.h -- transport-matrix products streamed without storing the plan
// ("FlashSinkhorn", Methodologie 3 and its HVP paragraph: the Hessian-vector
// product decomposes into transport-vector and transport-matrix products).
#pragma once
#include <cuda_runtime.h>

namespace sot {

// out[b][i][:] = sum_j P_ij V[b][j][:] with
// P_ij = w_i w'_j exp((fr_i + gc_j - |r_i - c_j|^2) / eps).
// Rows r (nr points) and columns c (nc points) are any two clouds of a
// problem: the f-side product uses (X, Y, f, g, a, b), the g-side product the
// same with the roles swapped.
struct TransportArgs {
    int B, nr, nc, d, c;
    const float* R;   // [B][nr][d] row points
    const float* Cl;  // [B][nc][d] column points
    const float* fr;  // [B][nr] row potentials
    const float* gc;  // [B][nc] column potentials
    const float* wr;  // [B][nr] row weights, NULL = uniform 1/nr
    const float* wc;  // [B][nc] column weights, NULL = uniform 1/nc
    const float* V;   // [B][nc] rows of c values, row stride ldv (>= c)
    float* out;       // [B][nr] rows of c values, row stride ldo (>= c)
    int ldv, ldo;
    float kap_hi, kap_lo;  // 1 / (eps ln 2) as a float-float pair
    int split, chunk;      // columns in `split` chunks of `chunk` columns (one CTA each)
    float* part;           // [split][B][nr][c] partial sums when split > 1
    const float* rc = nullptr;  // centred products: [B][nr][d] row barycentres
    const float* rv = nullptr;  // centred products: [B][nr][d] row directions
};

int transport_max_d();
int transport_max_c();
// Column split for a problem of d coordinates and c values per column on `sms`
// SMs (centred: the row-centred products, c = 1 with 2d values out per row):
// fills *split and *chunk; returns the floats of partial-sum scratch it needs
// (0 when split == 1).
size_t transport_plan(int B, int nr, int nc, int d, int c, bool centred, int sms, int* split, int* chunk);
cudaError_t launch_transport(const TransportArgs& p, cudaStream_t st);
cudaError_t launch_transport_centred(const TransportArgs& p, cudaStream_t st);
// g[k][j][:] <- 2 (w_j p_j - g[k][j][:]) for `count` points of d coordinates
// (w NULL = uniform 1/per_cloud): the gradient from the transport product.
cudaError_t launch_grad_finish(const float* P, const float* w, int B, int per_cloud, int d, float* g,
                               cudaStream_t st);

}  // namespace sot
