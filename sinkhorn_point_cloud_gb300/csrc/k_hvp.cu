// k_hvp.cu -- Hessian-vector product of the entropic OT loss with respect to X
// ("FlashSinkhorn", Methodologie 3, HVP paragraph: the product is built from
// transport-vector and transport-matrix products, never storing P).
//
// With P at the given potentials, r = P 1, c = P^T 1, moving X along V:
//   Cdot_ij = 2 (x_i - y_j) . v_i,
//   (fdot, gdot) keep both marginals: r_i fdot_i + (P gdot)_i = alpha_i,
//   (P^T fdot)_j + c_j gdot_j = beta_j (alpha, beta: row / column sums of P o Cdot).
// Eliminating fdot leaves S gdot = beta - P^T (alpha / r), S = diag(c) - P^T diag(1/r) P,
// solved by conjugate gradients preconditioned with diag(c), one system per cloud.
// The row constraint lets the assembly use the row barycentre yhat_i = (P Y)_i / r_i:
//   (H V)_i = 2 r_i v_i - (4/eps) sum_j P_ij ((y_j - yhat_i).v_i)(y_j - yhat_i)
//             - (2/eps) sum_j P_ij gdot_j (y_j - yhat_i),
// both sums formed pair by pair in the transport kernel's row-centred mode
// (the expanded second moments (P y y^T)_i v_i - yhat_i ((P Y)_i . v_i) cancel
// to a result |y|^2 / (eps / 2) times smaller than their terms).  The
// transport products run in the transport kernel; the kernels here pack their
// inputs, take the CG steps and assemble the result.
#include "common.cuh"
#include "hvp.h"
#include "kernels.h"

namespace sot {

constexpr int HV_T = 256;   // elementwise kernels
constexpr int HV_CG = 512;  // CG kernels: one block per cloud

template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        double t = (l < NT / 32) ? red[l] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    const double s = red[0];
    __syncthreads();  // red is reused by the next call
    return s;
}

__global__ void hvp_pack_ones_kernel(long long count, int d, const float* Y, float* A) {
    const long long j = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (j >= count) return;
    float* a = A + j * (1 + d);
    a[0] = 1.f;
    for (int k = 0; k < d; ++k) a[1 + k] = Y[j * d + k];
}

__global__ void hvp_pack_side1_kernel(long long count, int d, const float* X, const float* V, const float* PY1,
                                      float* W) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float* py = PY1 + i * (1 + d);
    const float r = py[0];
    float xv = 0.f, al = 0.f;
    for (int k = 0; k < d; ++k) {
        const float v = V[i * d + k];
        xv = fmaf(X[i * d + k], v, xv);
        al = fmaf(fmaf(r, X[i * d + k], -py[1 + k]), v, al);  // (r_i x_i - (P Y)_i) . v_i
    }
    float* w = W + i * (3 + d);
    w[0] = 1.f;
    w[1] = xv;
    w[2] = r > 0.f ? 2.f * al / r : 0.f;  // alpha_i / r_i
    for (int k = 0; k < d; ++k) w[3 + k] = V[i * d + k];
}

__global__ void hvp_rhs_kernel(long long count, int d, const float* Y, const float* PT, float* rhs, float* cvec) {
    const long long j = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (j >= count) return;
    const float* t = PT + j * (3 + d);
    float yv = 0.f;
    for (int k = 0; k < d; ++k) yv = fmaf(Y[j * d + k], t[3 + k], yv);
    cvec[j] = t[0];
    rhs[j] = 2.f * (t[1] - yv) - t[2];  // beta_j - (P^T alpha/r)_j
}

__global__ void __launch_bounds__(HV_CG) hvp_cg_init_kernel(int B, int m, const float* rhs, const float* cvec,
                                                            float* res, float* z, float* p, float* gd, HvpDots dots) {
    __shared__ double red[HV_CG / 32];
    const int b = blockIdx.x;
    const size_t o = (size_t)b * m;
    double s = 0.0;
    for (int j = threadIdx.x; j < m; j += HV_CG) {
        const float r = rhs[o + j], c = cvec[o + j];
        const float zz = c > 0.f ? r / c : 0.f;
        res[o + j] = r;
        z[o + j] = zz;
        p[o + j] = zz;
        gd[o + j] = 0.f;
        s += (double)r * zz;
    }
    s = block_sum_d<HV_CG>(s, red);
    if (threadIdx.x == 0) {
        dots.rz0[b] = s;
        dots.rz[b] = s;
    }
}

__global__ void hvp_div_r_kernel(long long count, int d, const float* Pp, const float* PY1, float* q) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float r = PY1[i * (1 + d)];
    q[i] = r > 0.f ? Pp[i] / r : 0.f;
}

// One CG step for cloud blockIdx.x, given Ptq = P^T ((P p) / r):
//   S p = c p - Ptq,  a = rz / (p . S p),  gd += a p,  res -= a S p,
//   z = res / c,  rz' = res . z,  p = z + (rz' / rz) p.
// A cloud whose preconditioned residual has fallen to tol^2 of its start (or
// whose p . S p is not positive) keeps its state.
__global__ void __launch_bounds__(HV_CG) hvp_cg_step_kernel(int B, int m, int it, float tol, const float* cvec,
                                                            const float* Ptq, float* p, float* Sp, float* res,
                                                            float* z, float* gd, HvpDots dots) {
    __shared__ double red[HV_CG / 32];
    const int b = blockIdx.x;
    const size_t o = (size_t)b * m;
    const double rzc = dots.rz[(size_t)(it & 1) * B + b];
    double* rzn = dots.rz + (size_t)((it + 1) & 1) * B + b;
    if (!(rzc > (double)tol * (double)tol * dots.rz0[b])) {
        if (threadIdx.x == 0) *rzn = rzc;
        return;
    }
    double s = 0.0;
    for (int j = threadIdx.x; j < m; j += HV_CG) {
        const float v = fmaf(cvec[o + j], p[o + j], -Ptq[o + j]);
        Sp[o + j] = v;
        s += (double)p[o + j] * v;
    }
    const double psp = block_sum_d<HV_CG>(s, red);
    if (!(psp > 0.0)) {
        if (threadIdx.x == 0) *rzn = 0.0;
        return;
    }
    const float a = (float)(rzc / psp);
    double s2 = 0.0;
    for (int j = threadIdx.x; j < m; j += HV_CG) {
        gd[o + j] = fmaf(a, p[o + j], gd[o + j]);
        const float r = fmaf(-a, Sp[o + j], res[o + j]);
        const float c = cvec[o + j];
        const float zz = c > 0.f ? r / c : 0.f;
        res[o + j] = r;
        z[o + j] = zz;
        s2 += (double)r * zz;
    }
    const double rz2 = block_sum_d<HV_CG>(s2, red);
    const float beta = (float)(rz2 / rzc);
    for (int j = threadIdx.x; j < m; j += HV_CG) p[o + j] = fmaf(beta, p[o + j], z[o + j]);
    if (threadIdx.x == 0) {
        *rzn = rz2;
        dots.psp[b] = psp;
    }
}

// Row barycentres yhat_i = (P Y)_i / r_i from PY1 [count][1+d] into YH [count][d].
__global__ void hvp_barycentre_kernel(long long count, int d, const float* PY1, float* YH) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float* py = PY1 + i * (1 + d);
    const float ir = py[0] > 0.f ? 1.f / py[0] : 0.f;
    for (int k = 0; k < d; ++k) YH[i * d + k] = py[1 + k] * ir;
}

// Assembly from the row-centred product CP [count][2d] = [r_i Cov_i v_i, sum_j P_ij g_j (y_j - yhat_i)]:
//   out_i = 2 r_i v_i - (4/eps) r_i Cov_i v_i - (2/eps) sum_j P_ij g_j (y_j - yhat_i).
__global__ void hvp_assemble_centred_kernel(long long count, int d, float eps, const float* V, const float* PY1,
                                            const float* CP, float* out) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float r = PY1[i * (1 + d)];
    const float* cp = CP + i * 2 * d;
    const float k4 = 4.f / eps, k2 = 2.f / eps;
    for (int k = 0; k < d; ++k) out[i * d + k] = 2.f * r * V[i * d + k] - k4 * cp[k] - k2 * cp[d + k];
}

static unsigned hv_blocks(long long count) { return (unsigned)((count + HV_T - 1) / HV_T); }

cudaError_t launch_hvp_pack_ones(long long count, int d, const float* Y, float* A, cudaStream_t st) {
    count_launches(1);
    hvp_pack_ones_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, Y, A);
    return cudaGetLastError();
}
cudaError_t launch_hvp_pack_side1(long long count, int d, const float* X, const float* V, const float* PY1,
                                  float* W, cudaStream_t st) {
    count_launches(1);
    hvp_pack_side1_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, X, V, PY1, W);
    return cudaGetLastError();
}
cudaError_t launch_hvp_rhs(long long count, int d, const float* Y, const float* PT, float* rhs, float* cvec,
                           cudaStream_t st) {
    count_launches(1);
    hvp_rhs_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, Y, PT, rhs, cvec);
    return cudaGetLastError();
}
cudaError_t launch_hvp_cg_init(int B, int m, const float* rhs, const float* cvec, float* res, float* z, float* p,
                               float* gd, HvpDots dots, cudaStream_t st) {
    count_launches(1);
    hvp_cg_init_kernel<<<B, HV_CG, 0, st>>>(B, m, rhs, cvec, res, z, p, gd, dots);
    return cudaGetLastError();
}
cudaError_t launch_hvp_div_r(long long count, int d, const float* Pp, const float* PY1, float* q, cudaStream_t st) {
    count_launches(1);
    hvp_div_r_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, Pp, PY1, q);
    return cudaGetLastError();
}
cudaError_t launch_hvp_cg_step(int B, int m, int it, float tol, const float* cvec, const float* Ptq, float* p,
                               float* Sp, float* res, float* z, float* gd, HvpDots dots, cudaStream_t st) {
    count_launches(1);
    hvp_cg_step_kernel<<<B, HV_CG, 0, st>>>(B, m, it, tol, cvec, Ptq, p, Sp, res, z, gd, dots);
    return cudaGetLastError();
}
cudaError_t launch_hvp_barycentre(long long count, int d, const float* PY1, float* YH, cudaStream_t st) {
    count_launches(1);
    hvp_barycentre_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, PY1, YH);
    return cudaGetLastError();
}
cudaError_t launch_hvp_assemble_centred(long long count, int d, float eps, const float* V, const float* PY1,
                                        const float* CP, float* out, cudaStream_t st) {
    count_launches(1);
    hvp_assemble_centred_kernel<<<hv_blocks(count), HV_T, 0, st>>>(count, d, eps, V, PY1, CP, out);
    return cudaGetLastError();
}

}  // namespace sot
