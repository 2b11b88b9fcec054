// k_apml.cu -- sparse APML on a stored COO support ("From Theory to
// Throughput: CUDA-Optimized APML", Abstract and Innovation).  With
// s_ij = -C_ij / T on the stored pairs:
//   row softmax R and column softmax K of s over the support,
//   P = (R + K) / 2 (bidirectional symmetrisation),
//   `iters` times: rows scaled to a, then columns scaled to b,
//   loss = sum P_ij C_ij.
// Row quantities are taken by one warp per row in a fixed order (the support
// is row-major, so a row is a contiguous range found from per-entry markers).
// Column sums add over a column's entries with fp64 atomics: their order
// varies, but fp64 sums of fp32 terms round to the same fp32 factor except in
// vanishingly rare ties.  An invalid support is flagged by the first pass and
// reported by the caller; every pass skips column indices out of range, so no
// pass touches memory outside its arrays in the meantime.
#include "apml.h"
#include "common.cuh"
#include "kernels.h"

namespace sot {

constexpr int AM_T = 256;

// Per entry: validation, C_ij (direct form), row range markers, column maxima of s.
__global__ void apml_prep_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const long long lo = p.off[b], hi = p.off[b + 1];
    if (hi < lo) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, SOT_DEV_BAD_COO);
        return;
    }
    const float* Xb = p.X + (size_t)b * p.n * p.d;
    const float* Yb = p.Y + (size_t)b * p.m * p.d;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = lo + blockIdx.x * (long long)blockDim.x + threadIdx.x; e < hi; e += stride) {
        const int i = p.rows[e], j = p.cols[e];
        if (i < 0 || i >= p.n || j < 0 || j >= p.m || (e + 1 < hi && p.rows[e + 1] < i)) {
            atomicOr(p.status, SOT_DEV_BAD_COO);
            continue;
        }
        const float* x = Xb + (size_t)i * p.d;
        const float* y = Yb + (size_t)j * p.d;
        float c = 0.f;
        for (int k = 0; k < p.d; ++k) {
            const float t = x[k] - y[k];
            c = fmaf(t, t, c);
        }
        p.cost[e] = c;
        // entries of row i are [rstart, rend) relative to the cloud's first entry + 1
        if (e == lo || p.rows[e - 1] != i) p.rstart[(size_t)b * p.n + i] = (int)(e - lo) + 1;
        if (e + 1 == hi || p.rows[e + 1] != i) p.rend[(size_t)b * p.n + i] = (int)(e - lo) + 1;
        atomicMax(p.cmax + (size_t)b * p.m + j, ord_encode(-c * p.inv_T));
    }
}

// Warp per row: row range (empty when no marker was written)
__device__ __forceinline__ bool apml_row_range(const ApmlArgs& p, int b, int i, long long* s0, long long* s1) {
    const int st = p.rstart[(size_t)b * p.n + i], en = p.rend[(size_t)b * p.n + i];
    if (st == 0) return false;
    *s0 = p.off[b] + st - 1;
    *s1 = p.off[b] + en;
    return true;
}

// Row softmax into vals; the column softmax's exponentials go to the column sums.
__global__ void apml_rowsoft_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * (AM_T / 32) + (threadIdx.x >> 5);
    if (i >= p.n) return;
    long long s0, s1;
    if (!apml_row_range(p, b, i, &s0, &s1)) return;
    float mx = -INFINITY;
    for (long long e = s0 + lane; e < s1; e += 32) mx = fmaxf(mx, -p.cost[e] * p.inv_T);
    mx = warp_max(mx);
    float sm = 0.f;
    for (long long e = s0 + lane; e < s1; e += 32) sm += expf(-p.cost[e] * p.inv_T - mx);
    sm = warp_sum(sm);
    for (long long e = s0 + lane; e < s1; e += 32) {
        const float s = -p.cost[e] * p.inv_T;
        p.vals[e] = expf(s - mx) / sm;
        const int j = p.cols[e];
        if (j < 0 || j >= p.m) continue;
        atomicAdd(p.csum + (size_t)b * p.m + j, (double)expf(s - ord_decode(p.cmax[(size_t)b * p.m + j])));
    }
}

// Per column, once: the fp32 factor the entries are scaled by (the fp64 pipe
// is slow here, so no entry pass converts or divides in fp64).
// mode 0: 1 / (column sum of the softmax exponentials); mode 1: b_j / (column sum).
__global__ void apml_colfactor_kernel(ApmlArgs p, int mode) {
    const long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (c >= (long long)p.B * p.m) return;
    const double cs = p.csum[c];
    if (mode == 0) {
        p.cfac[c] = cs > 0.0 ? (float)(1.0 / cs) : 0.f;
    } else {
        const double bj = p.b ? (double)p.b[c] : 1.0 / (double)p.m;
        p.cfac[c] = cs > 0.0 ? (float)(bj / cs) : 1.f;
    }
}

// P = (R + K) / 2 on every entry.
__global__ void apml_sym_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const long long lo = p.off[b], hi = p.off[b + 1];
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = lo + blockIdx.x * (long long)blockDim.x + threadIdx.x; e < hi; e += stride) {
        const int j = p.cols[e];
        if (j < 0 || j >= p.m) continue;
        const size_t cj = (size_t)b * p.m + j;
        const float k = expf(-p.cost[e] * p.inv_T - ord_decode(p.cmax[cj])) * p.cfac[cj];
        p.vals[e] = 0.5f * (p.vals[e] + k);
    }
}

// Rows scaled to a_i; the scaled values are added to the column sums.
__global__ void apml_rowscale_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * (AM_T / 32) + (threadIdx.x >> 5);
    if (i >= p.n) return;
    long long s0, s1;
    if (!apml_row_range(p, b, i, &s0, &s1)) return;
    float rs = 0.f;
    for (long long e = s0 + lane; e < s1; e += 32) rs += p.vals[e];
    rs = warp_sum(rs);
    const float ai = p.a ? p.a[(size_t)b * p.n + i] : 1.f / (float)p.n;
    const float f = rs > 0.f ? ai / rs : 1.f;
    for (long long e = s0 + lane; e < s1; e += 32) {
        const float v = p.vals[e] * f;
        p.vals[e] = v;
        const int j = p.cols[e];
        if (j >= 0 && j < p.m) atomicAdd(p.csum + (size_t)b * p.m + j, (double)v);
    }
}

// Columns scaled to b_j.
__global__ void apml_colscale_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const long long lo = p.off[b], hi = p.off[b + 1];
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = lo + blockIdx.x * (long long)blockDim.x + threadIdx.x; e < hi; e += stride) {
        const int j = p.cols[e];
        if (j < 0 || j >= p.m) continue;
        p.vals[e] *= p.cfac[(size_t)b * p.m + j];
    }
}

// Per-row loss terms sum_j P_ij C_ij (fixed order).
__global__ void apml_loss_kernel(ApmlArgs p) {
    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * (AM_T / 32) + (threadIdx.x >> 5);
    if (i >= p.n) return;
    long long s0 = 0, s1 = 0;
    float l = 0.f;
    if (apml_row_range(p, b, i, &s0, &s1))
        for (long long e = s0 + lane; e < s1; e += 32) l = fmaf(p.vals[e], p.cost[e], l);
    l = warp_sum(l);
    if (lane == 0) p.loss_part[(size_t)b * p.n + i] = l;
}

cudaError_t launch_apml(const ApmlArgs& p, cudaStream_t st) {
    if (p.B < 1 || p.n < 1 || p.m < 1 || p.d < 1 || !(p.inv_T > 0.f) || p.iters < 0) return cudaErrorInvalidValue;
    // per-entry passes: ~2048 blocks in all, so that every SM keeps enough loads
    // in flight (each thread's loop is a chain of dependent loads)
    const dim3 ge(2048 / p.B + 1, p.B), gr((p.n + AM_T / 32 - 1) / (AM_T / 32), p.B);
    const size_t csum_bytes = sizeof(double) * (size_t)p.B * p.m;
    count_launches(1);
    apml_prep_kernel<<<ge, AM_T, 0, st>>>(p);
    {
        cudaError_t e = cudaMemsetAsync(p.csum, 0, csum_bytes, st);
        if (e != cudaSuccess) return e;
    }
    const unsigned gf = (unsigned)(((long long)p.B * p.m + AM_T - 1) / AM_T);
    count_launches(1);
    apml_rowsoft_kernel<<<gr, AM_T, 0, st>>>(p);
    count_launches(1);
    apml_colfactor_kernel<<<gf, AM_T, 0, st>>>(p, 0);
    count_launches(1);
    apml_sym_kernel<<<ge, AM_T, 0, st>>>(p);
    for (int it = 0; it < p.iters; ++it) {
        cudaError_t e = cudaMemsetAsync(p.csum, 0, csum_bytes, st);
        if (e != cudaSuccess) return e;
        count_launches(1);
        apml_rowscale_kernel<<<gr, AM_T, 0, st>>>(p);
        count_launches(1);
        apml_colfactor_kernel<<<gf, AM_T, 0, st>>>(p, 1);
        count_launches(1);
        apml_colscale_kernel<<<ge, AM_T, 0, st>>>(p);
    }
    if (p.loss) {
        count_launches(1);
        apml_loss_kernel<<<gr, AM_T, 0, st>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_reduce_parts(p.loss_part, p.B, p.n, p.loss, st);
    }
    return cudaGetLastError();
}

}  // namespace sot
