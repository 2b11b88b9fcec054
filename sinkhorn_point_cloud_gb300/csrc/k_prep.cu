// k_prep.cu -- preprocessing and the small O(n) kernels around the fused
// half-steps: centring, packing, state <-> potential conversion, the stop
// decision, deterministic partial reductions, the COO scan and the gradient
// on a stored COO support.
#include "common.cuh"
#include "kernels.h"

namespace sot {

// ---- centring -------------------------------------------------------------
// shift[b][k] = (mean_i X[b][i][k] + mean_j Y[b][j][k]) / 2, accumulated in
// double in a fixed order.  C_ij is invariant under a common translation;
// centring shrinks |x|^2, |y|^2 and x.y and with them the rounding of the
// expanded-form score.
constexpr int CN_T = 256;
__global__ void __launch_bounds__(CN_T) center_kernel(const float* X, const float* Y, int n, int m, int d,
                                                      float* shift) {
    __shared__ double red[CN_T];
    const int b = blockIdx.y;
    const int k = blockIdx.x;  // one CTA per (coordinate, cloud)
    double sx = 0.0, sy = 0.0;
    const float* xb = X + (size_t)b * n * d;
    const float* yb = Y + (size_t)b * m * d;
    for (int i = threadIdx.x; i < n; i += CN_T) sx += (double)xb[(size_t)i * d + k];
    for (int j = threadIdx.x; j < m; j += CN_T) sy += (double)yb[(size_t)j * d + k];
    red[threadIdx.x] = sx / n + sy / m;
    __syncthreads();
    for (int s = CN_T / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) shift[(size_t)b * d + k] = (float)(0.5 * red[0]);
}

cudaError_t launch_center(const float* X, const float* Y, int B, int n, int m, int d, float* shift,
                          cudaStream_t st) {
    count_launches(1); center_kernel<<<dim3(d, B), CN_T, 0, st>>>(X, Y, n, m, d, shift);
    return cudaGetLastError();
}

// ---- packing --------------------------------------------------------------
// point layout (d <= 3): pack[b][i] = float4(x - t, log2 w) with zero padding;
// dense layout: pack[b][i][k] = x - t and lw2[b][i] = log2 w.
// nrm[b][i] = |x - t|^2 for the dense layout (expanded-form scores) and 0 for
// the point layout (direct-distance scores).  w == NULL means uniform weights 1/n.
__global__ void pack_kernel(const float* P, const float* w, int n, int d, const float* shift, int point,
                            float* pack, float* lw2, float* nrm) {
    const int b = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const size_t pi = (size_t)b * n + i;
    const float* src = P + pi * d;
    const float* sh = shift + (size_t)b * d;
    const float lw = w ? log2f(w[pi]) : -log2f((float)n);
    float acc = 0.f;
    if (point) {
        float v[3] = {0.f, 0.f, 0.f};
        for (int k = 0; k < d; ++k) {
            v[k] = src[k] - sh[k];
            acc = fmaf(v[k], v[k], acc);
        }
        reinterpret_cast<float4*>(pack)[pi] = make_float4(v[0], v[1], v[2], lw);
        acc = 0.f;  // the point path scores with direct distances: its state is L = -kappa f
    } else {
        float* dst = pack + pi * d;
        for (int k = 0; k < d; ++k) {
            const float v = src[k] - sh[k];
            dst[k] = v;
            acc = fmaf(v, v, acc);
        }
        lw2[pi] = lw;
    }
    nrm[pi] = acc;
}

cudaError_t launch_pack(const float* P, const float* w, int B, int n, int d, const float* shift, int point_layout,
                        float* pack, float* lw2, float* nrm, cudaStream_t st) {
    dim3 grid((n + 255) / 256, B);
    count_launches(1); pack_kernel<<<grid, 256, 0, st>>>(P, w, n, d, shift, point_layout, pack, lw2, nrm);
    return cudaGetLastError();
}

// ---- cosine cost -------------------------------------------------------------
// Unit directions: out[i] = P[i] / |P[i]| (a zero point stays zero).
__global__ void normalise_kernel(const float* P, long long count, int d, float* out) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float* s = P + i * d;
    float* o = out + i * d;
    float n2 = 0.f;
    for (int k = 0; k < d; ++k) n2 = fmaf(s[k], s[k], n2);
    const float nrm = sqrtf(n2);
    const float inv = nrm > 0.f ? 1.f / nrm : 0.f;
    for (int k = 0; k < d; ++k) o[k] = s[k] * inv;
}

cudaError_t launch_normalise(const float* P, long long count, int d, float* out, cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((count + 255) / 256);
    count_launches(1); normalise_kernel<<<blocks, 256, 0, st>>>(P, count, d, out);
    return cudaGetLastError();
}

// dst[i][k] = src[i][k] for k < d, 0 for d <= k < D (count points): a cloud
// at the tensor-core dimension D, whose extra coordinates add nothing.
__global__ void pad_kernel(const float* src, long long count, int d, int D, float* dst) {
    const long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (e >= count * D) return;
    const long long i = e / D;
    const int k = (int)(e - i * D);
    dst[e] = k < d ? src[i * d + k] : 0.f;
}

cudaError_t launch_pad(const float* src, long long count, int d, int D, float* dst, cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    const long long total = count * D;
    count_launches(1);
    pad_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(src, count, d, D, dst);
    return cudaGetLastError();
}

// grad_i <- (I - xhat_i xhat_i^T) grad_i / |x_i| (0 for a zero point): the
// gradient at the unit point xhat_i = x_i / |x_i| carried back to x_i.
__global__ void cosine_grad_kernel(const float* X, long long count, int d, float* grad) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= count) return;
    const float* x = X + i * d;
    float* gr = grad + i * d;
    float n2 = 0.f, dot = 0.f;
    for (int k = 0; k < d; ++k) {
        n2 = fmaf(x[k], x[k], n2);
        dot = fmaf(x[k], gr[k], dot);
    }
    if (!(n2 > 0.f)) {
        for (int k = 0; k < d; ++k) gr[k] = 0.f;
        return;
    }
    const float inv = 1.f / sqrtf(n2), c = dot / n2;
    for (int k = 0; k < d; ++k) gr[k] = (gr[k] - c * x[k]) * inv;
}

cudaError_t launch_cosine_grad(const float* X, long long count, int d, float* grad, cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((count + 255) / 256);
    count_launches(1); cosine_grad_kernel<<<blocks, 256, 0, st>>>(X, count, d, grad);
    return cudaGetLastError();
}

// ---- state <-> potential ----------------------------------------------------
// L = kappa (nrm - f);  f = nrm - L / kappa.
__global__ void state_from_pot_kernel(const float* nrm, const float* pot, float kappa, int count, float* state) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) state[i] = kappa * (nrm[i] - pot[i]);
}
__global__ void pot_from_state_kernel(const float* nrm, const float* state, float kappa, int count, float* pot) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) pot[i] = nrm[i] - state[i] / kappa;
}
// Cold start (f = g = 0): state = kappa * nrm.
__global__ void state_cold_kernel(const float* nrm, float kappa, int count, float* state) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) state[i] = kappa * nrm[i];
}
__global__ void scale_kernel(float* v, float s, int count) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) v[i] *= s;
}
__global__ void copy_kernel(float* dst, const float* src, int count, const int* stop_flag) {
    if (stop_flag && *(volatile const int*)stop_flag) return;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) dst[i] = src[i];
}

cudaError_t launch_state_from_potential(const float* nrm, const float* pot, float kappa, int count, float* state,
                                        cudaStream_t st) {
    count_launches(1); state_from_pot_kernel<<<(count + 255) / 256, 256, 0, st>>>(nrm, pot, kappa, count, state);
    return cudaGetLastError();
}
cudaError_t launch_potential_from_state(const float* nrm, const float* state, float kappa, int count, float* pot,
                                        cudaStream_t st) {
    count_launches(1); pot_from_state_kernel<<<(count + 255) / 256, 256, 0, st>>>(nrm, state, kappa, count, pot);
    return cudaGetLastError();
}
cudaError_t launch_state_cold(const float* nrm, float kappa, int count, float* state, cudaStream_t st) {
    count_launches(1); state_cold_kernel<<<(count + 255) / 256, 256, 0, st>>>(nrm, kappa, count, state);
    return cudaGetLastError();
}
cudaError_t launch_scale(float* v, float s, int count, cudaStream_t st) {
    count_launches(1); scale_kernel<<<(count + 255) / 256, 256, 0, st>>>(v, s, count);
    return cudaGetLastError();
}
cudaError_t launch_copy(float* dst, const float* src, int count, const int* stop_flag, cudaStream_t st) {
    count_launches(1); copy_kernel<<<(count + 255) / 256, 256, 0, st>>>(dst, src, count, stop_flag);
    return cudaGetLastError();
}

// ---- deterministic partial sums: out[b] = sum_p part[b][p] ------------------
__global__ void reduce_parts_kernel(const float* part, int parts, float* out) {
    __shared__ float red[8];
    const int b = blockIdx.x;
    float s = 0.f;
    for (int p = threadIdx.x; p < parts; p += 256) s += part[(size_t)b * parts + p];
    s = block_sum<256>(s, red);
    if (threadIdx.x == 0) out[b] = s;
}
cudaError_t launch_reduce_parts(const float* part, int B, int parts, float* out, cudaStream_t st) {
    count_launches(1); reduce_parts_kernel<<<B, 256, 0, st>>>(part, parts, out);
    return cudaGetLastError();
}

// ---- stop decision ----------------------------------------------------------
// One CTA.  err[b] = sum_p errpart[b][p]; if max_b err[b] < tol (or force):
// *stop_flag = 1 (the committed state stays the previous iterate), *conv_flag
// records a pass of the test; otherwise the tested half-step is committed by
// copying L_next -> L_cur.  Does nothing if the stage already stopped.
__global__ void decide_kernel(const float* errpart, int B, int parts, float tol, int force_stop, float* err_out,
                              int* stop_flag, int* conv_flag, const float* L_next, float* L_cur, int count) {
    __shared__ float red[8];
    __shared__ int s_stop;
    if (*(volatile int*)stop_flag) return;
    float emax = 0.f;
    for (int b = 0; b < B; ++b) {
        float s = 0.f;
        for (int p = threadIdx.x; p < parts; p += 256) s += errpart[(size_t)b * parts + p];
        s = block_sum<256>(s, red);
        if (threadIdx.x == 0 && err_out) err_out[b] = s;
        emax = fmaxf(emax, s);
    }
    if (threadIdx.x == 0) {
        const int pass = emax < tol;  // NaN fails
        s_stop = pass || force_stop;
        if (pass && conv_flag) *conv_flag = 1;
    }
    __syncthreads();
    if (s_stop) {
        __syncthreads();
        if (threadIdx.x == 0) *stop_flag = 1;
        return;
    }
    for (int i = threadIdx.x; i < count; i += 256) L_cur[i] = L_next[i];
}
cudaError_t launch_decide(const float* errpart, int B, int parts, float tol, int force_stop, float* err_out,
                          int* stop_flag, int* conv_flag, const float* L_next, float* L_cur, int count,
                          cudaStream_t st) {
    count_launches(1); decide_kernel<<<1, 256, 0, st>>>(errpart, B, parts, tol, force_stop, err_out, stop_flag, conv_flag, L_next,
                                     L_cur, count);
    return cudaGetLastError();
}

// counter += 1 unless the stage has stopped (counts realised iterations).
__global__ void count_iter_kernel(const int* stop_flag, int* counter) {
    if (stop_flag && *(volatile const int*)stop_flag) return;
    *counter += 1;
}
cudaError_t launch_count_iter(const int* stop_flag, int* counter, cudaStream_t st) {
    count_launches(1); count_iter_kernel<<<1, 1, 0, st>>>(stop_flag, counter);
    return cudaGetLastError();
}

// ---- device status of asynchronous calls -------------------------------------
// Bits of the per-call status words of asynchronous calls, gathered per device
// until the host reads and clears them (sot_async_status).
__device__ unsigned g_async_status;

__global__ void status_merge_kernel(const int* status) { atomicOr(&g_async_status, (unsigned)*status); }
cudaError_t launch_status_merge(const int* status, cudaStream_t st) {
    count_launches(1); status_merge_kernel<<<1, 1, 0, st>>>(status);
    return cudaGetLastError();
}
cudaError_t read_clear_async_status(cudaStream_t st, unsigned* out) {
    unsigned v = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_async_status, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_async_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    *out = v;
    return e;
}

// ---- input validation ---------------------------------------------------------
__global__ void check_kernel(const float* X, long long npts, const float* w, long long nw, int* bad) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < npts; e += stride)
        if (!isfinite(X[e])) atomicOr(bad, 1);
    if (w)
        for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < nw; e += stride)
            if (!(isfinite(w[e]) && w[e] > 0.f)) atomicOr(bad, 2);
}
cudaError_t launch_check_inputs(const float* X, const float* w, long long count_pts, int d, long long count_w,
                                int* bad, cudaStream_t st) {
    count_launches(1); check_kernel<<<256, 256, 0, st>>>(X, count_pts * d, w, count_w, bad);
    return cudaGetLastError();
}

// ---- COO scan -----------------------------------------------------------------
// rowptr[k] = sum_{k' < k} counts[k'] over all B*n rows (cloud after cloud),
// batch_offsets[b] = rowptr[b n], batch_offsets[B] = rowptr[B n] = nnz.
constexpr int SC_T = 1024;
__global__ void __launch_bounds__(SC_T) scan_kernel(const int* counts, int B, int n, long long* rowptr,
                                                    long long* batch_offsets) {
    __shared__ long long part[SC_T];
    const long long total = (long long)B * n;
    const long long seg = (total + SC_T - 1) / SC_T;
    const long long lo = threadIdx.x * seg, hi = min(total, lo + seg);
    long long s = 0;
    for (long long k = lo; k < hi; ++k) s += counts[k];
    part[threadIdx.x] = s;
    __syncthreads();
    // Hillis-Steele inclusive scan of the segment sums
    for (int o = 1; o < SC_T; o <<= 1) {
        long long v = (threadIdx.x >= o) ? part[threadIdx.x - o] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    long long run = (threadIdx.x == 0) ? 0 : part[threadIdx.x - 1];
    for (long long k = lo; k < hi; ++k) {
        rowptr[k] = run;
        run += counts[k];
    }
    if (threadIdx.x == SC_T - 1) rowptr[total] = part[SC_T - 1];
    __syncthreads();
    for (int b = threadIdx.x; b <= B; b += SC_T) batch_offsets[b] = rowptr[(long long)b * n];
}
cudaError_t launch_scan_counts(const int* counts, int B, int n, long long* rowptr, long long* batch_offsets,
                               cudaStream_t st) {
    count_launches(1); scan_kernel<<<1, SC_T, 0, st>>>(counts, B, n, rowptr, batch_offsets);
    return cudaGetLastError();
}

// ---- gradient on a stored support ------------------------------------------------
// grad[b][i] = 2 sum_{e: rows[e] = i} vals[e] (x_i - y_cols[e]).  One warp per
// row; the row's segment of the row-sorted COO is found by binary search;
// lanes walk the coordinates (d > 3) or the entries (d <= 3) and the sums are
// taken in entry order, so the result is deterministic.  Entries whose column
// is out of range are skipped and flagged; unsorted input is flagged by the
// validation pass.
__global__ void coo_validate_kernel(const int* rows, const int* cols, const long long* off, int n, int m,
                                    int* status) {
    const int b = blockIdx.y;
    const long long lo = off[b], hi = off[b + 1];
    if (hi < lo) { if (threadIdx.x == 0) atomicOr(status, SOT_DEV_BAD_COO); return; }
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = lo + blockIdx.x * (long long)blockDim.x + threadIdx.x; e < hi; e += stride) {
        const int i = rows[e], j = cols[e];
        bool bad = i < 0 || i >= n || j < 0 || j >= m;
        if (e + 1 < hi && rows[e + 1] < i) bad = true;
        if (bad) atomicOr(status, SOT_DEV_BAD_COO);
    }
}

// First e in [lo, hi) with rows[e] >= key (hi if none), rows sorted ascending;
// the whole warp searches together: 32 probes per round cut the range ~33-fold,
// so a round trip to memory is paid log_33 of the range times, not log_2.
__device__ __forceinline__ long long warp_lower_bound_rows(const int* rows, long long lo, long long hi, int key) {
    const int lane = threadIdx.x & 31;
    while (hi - lo > 32) {  // invariant: the answer lies in [lo, hi]
        const long long step = (hi - lo + 32) / 33;
        const long long pos = lo + step * (lane + 1) - 1;
        const int c = __popc(__ballot_sync(0xffffffffu, pos < hi && rows[pos] < key));
        const long long nlo = lo + step * c;
        const long long nhi = (c == 32) ? hi : lo + step * (c + 1) - 1;
        lo = nlo;
        hi = nhi < hi ? nhi : hi;
    }
    const long long pos = lo + lane;
    return lo + __popc(__ballot_sync(0xffffffffu, pos < hi && rows[pos] < key));
}

__global__ void grad_coo_kernel(const float* X, const float* Y, int n, int m, int d, const int* rows,
                                const int* cols, const float* vals, const long long* off, float* grad,
                                int* status) {
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * (blockDim.x >> 5) + warp;
    if (i >= n) return;
    const long long lo = off[b], hi = off[b + 1];
    const long long s0 = warp_lower_bound_rows(rows, lo, hi, i);
    const long long s1 = warp_lower_bound_rows(rows, s0, hi, i + 1);
    const float* xi = X + ((size_t)b * n + i) * d;
    const float* yb = Y + (size_t)b * m * d;
    float* gi = grad + ((size_t)b * n + i) * d;
    if (d <= 3) {
        float g0 = 0.f, g1 = 0.f, g2 = 0.f;
        for (long long e = s0 + lane; e < s1; e += 32) {
            const int j = cols[e];
            if (j < 0 || j >= m || rows[e] != i) { atomicOr(status, SOT_DEV_BAD_COO); continue; }
            const float v = vals[e];
            const float* y = yb + (size_t)j * d;
            g0 = fmaf(v, xi[0] - y[0], g0);
            if (d > 1) g1 = fmaf(v, xi[1] - y[1], g1);
            if (d > 2) g2 = fmaf(v, xi[2] - y[2], g2);
        }
        g0 = warp_sum(g0); g1 = warp_sum(g1); g2 = warp_sum(g2);
        if (lane == 0) {
            gi[0] = 2.f * g0;
            if (d > 1) gi[1] = 2.f * g1;
            if (d > 2) gi[2] = 2.f * g2;
        }
    } else {
        for (int k0 = 0; k0 < d; k0 += 32) {
            const int k = k0 + lane;
            float g = 0.f;
            for (long long e = s0; e < s1; ++e) {
                const int j = cols[e];
                if (j < 0 || j >= m) { if (lane == 0 && k0 == 0) atomicOr(status, SOT_DEV_BAD_COO); continue; }
                if (k < d) g = fmaf(vals[e], xi[k] - yb[(size_t)j * d + k], g);
            }
            if (k < d) gi[k] = 2.f * g;
        }
    }
}

cudaError_t launch_grad_coo(const float* X, const float* Y, int B, int n, int m, int d, const int* rows,
                            const int* cols, const float* vals, const long long* batch_offsets, float* grad,
                            int* status, cudaStream_t st) {
    count_launches(1); coo_validate_kernel<<<dim3(4 * 152 / (B > 0 ? B : 1) + 1, B), 256, 0, st>>>(rows, cols, batch_offsets, n, m, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1); grad_coo_kernel<<<dim3((n + 7) / 8, B), 256, 0, st>>>(X, Y, n, m, d, rows, cols, vals, batch_offsets, grad,
                                                           status);
    return cudaGetLastError();
}

}  // namespace sot
