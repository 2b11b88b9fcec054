// hvp.h -- Hessian-vector product of the entropic OT loss with respect to X
// ("FlashSinkhorn", Methodologie 3, HVP paragraph) from transport products.
#pragma once
#include <cuda_runtime.h>

namespace sot {

// Largest d: the row-centred product keeps 3 d values per row in registers.
constexpr int HVP_MAX_D = 9;

// Per-cloud conjugate-gradient scalars (fp64), 4 B values in all.
struct HvpDots {
    double* rz0;  // initial preconditioned residual
    double* rz;   // [2][B] current / next preconditioned residual
    double* psp;  // p . S p
};

// [B*m][1 + d]: 1, y_j
cudaError_t launch_hvp_pack_ones(long long count, int d, const float* Y, float* A, cudaStream_t st);
// rows i of P [1, Y] (PY1 [B*n][1+d]) and V -> W [B*n][3+d]: 1, x.v, alpha/r, v
cudaError_t launch_hvp_pack_side1(long long count, int d, const float* X, const float* V, const float* PY1,
                                  float* W, cudaStream_t st);
// columns j of P^T W (PT [B*m][3+d]) -> rhs_j = beta_j - (P^T alpha/r)_j and c_j
cudaError_t launch_hvp_rhs(long long count, int d, const float* Y, const float* PT, float* rhs, float* cvec,
                           cudaStream_t st);
// CG steps on S = diag(c) - P^T diag(1/r) P, one system per cloud
cudaError_t launch_hvp_cg_init(int B, int m, const float* rhs, const float* cvec, float* res, float* z, float* p,
                               float* gd, HvpDots dots, cudaStream_t st);
cudaError_t launch_hvp_div_r(long long count, int d, const float* Pp, const float* PY1, float* q, cudaStream_t st);
cudaError_t launch_hvp_cg_step(int B, int m, int it, float tol, const float* cvec, const float* Ptq, float* p,
                               float* Sp, float* res, float* z, float* gd, HvpDots dots, cudaStream_t st);
// Row-centred assembly (the accurate route): yhat = (P Y) / r, then the centred
// product CP [B*n][2d] of g' (see launch_transport_centred) and
// out_i = 2 r_i v_i - (4/eps) CP_i[0:d] - (2/eps) CP_i[d:2d].
cudaError_t launch_hvp_barycentre(long long count, int d, const float* PY1, float* YH, cudaStream_t st);
cudaError_t launch_hvp_assemble_centred(long long count, int d, float eps, const float* V, const float* PY1,
                                        const float* CP, float* out, cudaStream_t st);

}  // namespace sot
