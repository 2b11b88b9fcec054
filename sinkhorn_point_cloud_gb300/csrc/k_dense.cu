// k_dense.cu -- fp32 FMA Sinkhorn kernels for any dimension d <= 1024.
//
// This is the full-precision path for d > 3 (SOT_PREC_FP32, and dimensions
// the tensor-core path does not take).  Same fused half-step as the point
// path ("FlashSinkhorn", Methodologie 1-2): a 64-row block stays resident in
// shared memory while 64-column tiles stream past; each thread forms a 4 x 4
// micro-tile of dot products in registers, turns it into scores, and the row
// log-sum-exp is reduced across the 16 threads that share a row with
// shuffles.  Nothing of size n x m is written.  Above d = 256 ("FlashSinkhorn",
// Experimentele Resultaten: d up to 1024) the coordinates stream in slices of
// 256: the row block's slice is staged again with each column tile's, and the
// dot products carry on across the slices in the same k-ascending order.
#include "common.cuh"
#include "kernels.h"

namespace sot {

constexpr int DN_T = 256;
constexpr int DN_RT = 64;    // rows per CTA
constexpr int DN_CT = 64;    // columns per tile
constexpr int DN_DK = 256;   // coordinates per shared-memory slice
constexpr int DN_MAXD = 1024;

int dense_rows_per_cta() { return DN_RT; }
int dense_cols_per_tile() { return DN_CT; }
int dense_max_d() { return DN_MAXD; }

__host__ __device__ inline int dense_dk(int d) { return d < DN_DK ? d : DN_DK; }

// Shared memory holds the staged slices k-major: coordinate k of row r at
// k * DN_LDT + r, so that a thread's four rows (and four columns) at one k are
// one 16-byte read.  Xs[dk][DN_LDT], Ys[dk][DN_LDT] with dk = min(d, 256), then
// cs[DN_CT] column bias.
constexpr int DN_LDT = DN_RT + 4;
static_assert(DN_RT == DN_CT && DN_LDT % 4 == 0, "k-major tiles");
__host__ __device__ inline size_t dense_smem_bytes(int d) {
    return sizeof(float) * ((size_t)2 * dense_dk(d) * DN_LDT + DN_CT + DN_T / 32 + 8);
}

// acc[rr][cc] += sum_k x[4tr+rr][k] * y[4tc+cc][k] over the kw coordinates of
// a staged slice, k ascending, fp32 FMA.
__device__ __forceinline__ void dense_dot_tile(const float* Xs, const float* Ys, int kw, int tr, int tc,
                                               float acc[4][4]) {
    const float4* xp = reinterpret_cast<const float4*>(Xs) + tr;
    const float4* yp = reinterpret_cast<const float4*>(Ys) + tc;
#pragma unroll 4
    for (int k = 0; k < kw; ++k) {
        const float4 x4 = xp[k * (DN_LDT / 4)], y4 = yp[k * (DN_LDT / 4)];
        const float xv[4] = {x4.x, x4.y, x4.z, x4.w}, yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc[rr][cc] = fmaf(xv[rr], yv[cc], acc[rr][cc]);
    }
}

__device__ __forceinline__ void zero_tile(float acc[4][4]) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) acc[rr][cc] = 0.f;
}

__device__ __forceinline__ float sum16(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float max16(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Copy coordinates [k0, k0 + kw) of `cnt` rows (row-major [*][d]) starting at
// `row0` into the k-major S[kw][DN_LDT], zero-filling rows past `lim`.
__device__ __forceinline__ void dense_stage(float* S, const float* src, int row0, int cnt, int lim, int d, int k0,
                                            int kw) {
    for (int e = threadIdx.x; e < cnt * kw; e += DN_T) {
        const int r = e / kw, k = e - r * kw;
        const int gr = row0 + r;
        S[k * DN_LDT + r] = (gr < lim) ? src[(size_t)gr * d + k0 + k] : 0.f;
    }
}

// acc = the row block's dot products with column tile [base, base + DN_CT):
// for d <= 256 the row block is staged once by the caller (Xs) and only the
// column tile is staged here; above, both are staged slice by slice.
// `cols_bias` runs with the first slice's staging, before its barrier.  On
// return the last slice is still staged.
template <class Bias>
__device__ __forceinline__ void dense_tile_dots(float* Xs, float* Ys, const float* rows, const float* cols, int row0,
                                                int nr, int base, int c_end, int d, int tr, int tc, float acc[4][4],
                                                Bias&& cols_bias) {
    const int dk = dense_dk(d);
    zero_tile(acc);
    for (int k0 = 0; k0 < d; k0 += dk) {
        const int kw = min(dk, d - k0);
        __syncthreads();  // the previous slice (or tile) is no longer read
        if (d > dk) dense_stage(Xs, rows, row0, DN_RT, nr, d, k0, kw);
        dense_stage(Ys, cols, base, DN_CT, c_end, d, k0, kw);
        if (k0 == 0) cols_bias();
        __syncthreads();
        dense_dot_tile(Xs, Ys, kw, tr, tc, acc);
    }
}

// Dot product of one row with one column straight from global memory (slow paths).
__device__ __forceinline__ float dense_dot_global(const float* x, const float* y, int d) {
    float acc = 0.f;
    for (int k = 0; k < d; ++k) acc = fmaf(x[k], y[k], acc);
    return acc;
}

template <int MODE>
__global__ void __launch_bounds__(DN_T) dense_half_kernel(HalfArgs p) {
    if (p.stop_flag && *(volatile const int*)p.stop_flag) return;
    extern __shared__ float smem[];
    const int d = p.d, dk = dense_dk(d);
    float* Xs = smem;
    float* Ys = Xs + dk * DN_LDT;
    float* cs = Ys + dk * DN_LDT;
    float* red = cs + DN_CT;
    int* flags = reinterpret_cast<int*>(red + DN_T / 32);  // [0] last, [1] nretry

    const int b = blockIdx.y;
    const int rt = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rt * DN_RT;
    const int c_begin = ch * p.chunk, c_end = min(p.nc, c_begin + p.chunk);
    const float* rows = p.rpack + (size_t)b * p.nr * d;
    const float* cols = p.cpack + (size_t)b * p.nc * d;
    const float* cw = p.cw2 + (size_t)b * p.nc;
    const float* cst = p.cstate + (size_t)b * p.nc;
    const size_t rbase = (size_t)b * p.nr;
    const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;

    if (p.lo_reset && blockIdx.x == 0 && blockIdx.y == 0)
        for (int k = threadIdx.x; k < p.B; k += DN_T) p.lo_reset[k] = SOT_ORD_EMPTY;
    if (d <= DN_DK) dense_stage(Xs, rows, row0, DN_RT, p.nr, d, 0, d);
    float m[4], s[4], old[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int row = row0 + 4 * tr + rr;
        old[rr] = (MODE == MODE_LSE && row < p.nr && p.rstate_in) ? p.rstate_in[rbase + row] : 0.f;
        if (MODE == MODE_MAX) m[rr] = -INFINITY;
        else if (row >= p.nr) m[rr] = INFINITY;
        else m[rr] = stabiliser(p.cold, p.lo_in, b, old[rr]);
        s[rr] = 0.f;
    }
    const float tk = p.two_kappa;

    for (int base = c_begin; base < c_end; base += DN_CT) {
        float acc[4][4];
        dense_tile_dots(Xs, Ys, rows, cols, row0, p.nr, base, c_end, d, tr, tc, acc, [&] {
            for (int c = threadIdx.x; c < DN_CT; c += DN_T) {
                const int j = base + c;
                cs[c] = (j < c_end) ? cw[j] - cst[j] : -INFINITY;
            }
        });
        float cb[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) cb[cc] = cs[4 * tc + cc];
        if (MODE == MODE_MAX) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                float mx = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) mx = fmaxf(mx, fmaf(tk, acc[rr][cc], cb[cc]));
                m[rr] = fmaxf(m[rr], max16(mx));
            }
        } else {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                float ts = 0.f;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) ts += ex2f(fmaf(tk, acc[rr][cc], cb[cc] - m[rr]));
                ts = sum16(ts);
                // The two half-warps own different rows: the slow path is entered by
                // the whole warp (its shuffles need every lane) and applied per row.
                const bool ovf = !(ts < SOT_TILE_SUM_MAX);
                if (__any_sync(0xffffffffu, ovf)) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) mx = fmaxf(mx, fmaf(tk, acc[rr][cc], cb[cc]));
                    mx = max16(mx);
                    const float mn = fmaxf(m[rr], mx);
                    const float mu = (ovf && mn > -INFINITY) ? mn : m[rr];
                    float ts2 = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) ts2 += ex2f(fmaf(tk, acc[rr][cc], cb[cc] - mu));
                    ts2 = sum16(ts2);
                    if (ovf) {
                        if (mn == -INFINITY) {
                            ts = 0.f;
                        } else {
                            s[rr] = (m[rr] == -INFINITY) ? 0.f : s[rr] * ex2f(m[rr] - mn);
                            m[rr] = mn;
                            ts = ts2;
                        }
                    }
                }
                s[rr] += ts;
            }
        }
    }

    // ---- combine column chunks (thread tc == 0 of each row group owns its rows) ----
    if (p.split > 1) {
        const size_t stride = (size_t)p.B * p.nr;
        if (tc == 0) {
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int row = row0 + 4 * tr + rr;
                if (row < p.nr) {
                    p.part_m[ch * stride + rbase + row] = m[rr];
                    if (MODE == MODE_LSE) p.part_s[ch * stride + rbase + row] = s[rr];
                }
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned prev = atomicAdd(&p.counters[b * p.rowtiles + rt], 1u);
            flags[0] = (prev == (unsigned)(p.split - 1));
        }
        __syncthreads();
        if (!flags[0]) return;
        __threadfence();
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = row0 + 4 * tr + rr;
            float M = -INFINITY, S = 0.f;
            if (row < p.nr) {
                for (int c = 0; c < p.split; ++c) {
                    const float pm = __ldcg(p.part_m + c * stride + rbase + row);
                    if (MODE == MODE_MAX) M = fmaxf(M, pm);
                    else lse_combine(M, S, pm, __ldcg(p.part_s + c * stride + rbase + row));
                }
            }
            m[rr] = M;
            s[rr] = S;
        }
        if (threadIdx.x == 0) p.counters[b * p.rowtiles + rt] = 0u;
    }

    // ---- finalise ---------------------------------------------------------
    int* retry_rows = reinterpret_cast<int*>(Ys);  // reuse the column tile buffer
    if (threadIdx.x == 0) flags[1] = 0;
    __syncthreads();
    if (tc == 0) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int row = row0 + 4 * tr + rr;
            if (row >= p.nr) continue;
            if (MODE == MODE_MAX) p.rstate_out[rbase + row] = m[rr];
            else if (s[rr] >= SOT_SUM_MIN && s[rr] < INFINITY && m[rr] > -INFINITY)
                p.rstate_out[rbase + row] = m[rr] + log2f(s[rr]);
            else retry_rows[atomicAdd(&flags[1], 1)] = row;
        }
    }
    __syncthreads();
    if (MODE == MODE_LSE) {
        const int nretry = flags[1];
        for (int k = 0; k < nretry; ++k) {
            const int row = retry_rows[k];
            const float* xr = rows + (size_t)row * d;
            float mx = -INFINITY;
            for (int j = threadIdx.x; j < p.nc; j += DN_T)
                mx = fmaxf(mx, fmaf(tk, dense_dot_global(xr, cols + (size_t)j * d, d), cw[j] - cst[j]));
            mx = block_max<DN_T>(mx, red);
            float sm = 0.f;
            if (mx > -INFINITY)
                for (int j = threadIdx.x; j < p.nc; j += DN_T)
                    sm += ex2f(fmaf(tk, dense_dot_global(xr, cols + (size_t)j * d, d), cw[j] - cst[j]) - mx);
            sm = block_sum<DN_T>(sm, red);
            if (threadIdx.x == 0) {
                p.rstate_out[rbase + row] = (mx > -INFINITY) ? mx + log2f(sm) : -INFINITY;
                atomicOr(p.status, SOT_DEV_RETRY_ROWS);
            }
        }
        if (p.errpart || p.lo_out) {
            __syncthreads();
            float e = 0.f, lo = INFINITY;
            const float wu = 1.f / (float)p.nr;
            if (tc == 0) {
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int row = row0 + 4 * tr + rr;
                    if (row >= p.nr) continue;
                    const float nv = p.rstate_out[rbase + row];
                    const float w = p.rweight ? p.rweight[rbase + row] : wu;
                    e += w * fabsf(ex2f(nv - old[rr]) - 1.f);
                    lo = fminf(lo, old[rr] - nv);
                }
            }
            if (p.errpart) {
                e = block_sum<DN_T>(e, red);
                if (threadIdx.x == 0) p.errpart[b * p.rowtiles + rt] = e;
            }
            if (p.lo_out) {
                lo = warp_min(lo);
                if ((threadIdx.x & 31) == 0 && lo < INFINITY) atomicMin(p.lo_out + b, ord_encode(lo));
            }
        }
    }
}

cudaError_t launch_dense_half(const HalfArgs& p, int mode, cudaStream_t st) {
    if (p.d < 1 || p.d > DN_MAXD) return cudaErrorInvalidValue;
    const size_t sm = dense_smem_bytes(p.d);
    dim3 grid(p.rowtiles * p.split, p.B), block(DN_T);
    cudaError_t e;
    if (mode == MODE_MAX) {
        e = cudaFuncSetAttribute(dense_half_kernel<MODE_MAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        count_launches(1); dense_half_kernel<MODE_MAX><<<grid, block, sm, st>>>(p);
    } else {
        e = cudaFuncSetAttribute(dense_half_kernel<MODE_LSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        count_launches(1); dense_half_kernel<MODE_LSE><<<grid, block, sm, st>>>(p);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Plan application, dense ("FlashSinkhorn", Methodologie 3).  P_ij / a_i =
// 2^(2 kappa x_i.y_j + log2 b_j - Lam_j - L_i) (the f-half score against the
// final row value); C_ij = nx_i + ny_j - 2 x_i.y_j.  After the scores of a
// tile are exponentiated, P goes to shared memory and a second in-smem product
// accumulates v_i = sum_j P_ij y_j, each thread owning 4 rows x KV coordinates.
template <int KV>
__global__ void __launch_bounds__(DN_T) dense_apply_kernel(ApplyArgs p) {
    extern __shared__ float smem[];
    const int d = p.d, dk = dense_dk(d);
    float* Xs = smem;
    float* Ys = Xs + dk * DN_LDT;
    float* cs = Ys + dk * DN_LDT;
    float* red = cs + DN_CT;
    float* Ps = red + DN_T / 32 + 8;  // [DN_RT][DN_CT + 1]
    float* nys = Ps + DN_RT * (DN_CT + 1);
    const int b = blockIdx.y;
    const int row0 = blockIdx.x * DN_RT;
    // coordinates [kb0, kb0 + kwz) of the gradient (blockIdx.z: one slice of 256 each above d = 256)
    const int kb0 = blockIdx.z * dk, kwz = min(dk, d - kb0);
    const float* rows = p.xpack + (size_t)b * p.n * d;
    const float* cols = p.ypack + (size_t)b * p.m * d;
    const size_t xb = (size_t)b * p.n, yb = (size_t)b * p.m;
    const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;
    const float tk = 2.f * p.kappa;
    const float kh = (float)p.kappa64;
    const float2 kap = make_float2(kh, (float)(p.kappa64 - (double)kh));
    const float sig_thr = -(30.f + log2f((float)p.m));

    if (d <= DN_DK) dense_stage(Xs, rows, row0, DN_RT, p.n, d, 0, d);
    float Lr[4], nxr[4], m[4], r_[4], q_[4], v[4][KV];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int row = row0 + 4 * tr + rr;
        const bool ok = row < p.n;
        Lr[rr] = ok ? p.L[xb + row] : 0.f;
        nxr[rr] = ok ? p.nx[xb + row] : 0.f;
        m[rr] = ok ? -SOT_STAB_BIAS : INFINITY;
        r_[rr] = q_[rr] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KV; ++kk) v[rr][kk] = 0.f;
    }
    for (int base = 0; base < p.m; base += DN_CT) {
        float acc[4][4];
        dense_tile_dots(Xs, Ys, rows, cols, row0, p.n, base, p.m, d, tr, tc, acc, [&] {
            for (int c = threadIdx.x; c < DN_CT; c += DN_T) {
                const int j = base + c;
                cs[c] = (j < p.m) ? p.lw2y[yb + j] - p.Lam[yb + j] : -INFINITY;
                nys[c] = (j < p.m) ? p.ny[yb + j] : 0.f;
            }
        });
        float cb[4], nyc[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) { cb[cc] = cs[4 * tc + cc]; nyc[cc] = nys[4 * tc + cc]; }
        float sc[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            // exponent relative to the row stabiliser: score - L_i - m
            float w[4], ts = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                w[cc] = ex2f(fmaf(tk, acc[rr][cc], cb[cc] - Lr[rr] - m[rr]));
                ts += w[cc];
            }
            ts = sum16(ts);
            sc[rr] = 1.f;
            const bool ovf = !(ts < SOT_TILE_SUM_MAX);
            if (__any_sync(0xffffffffu, ovf)) {  // warp-wide: the shuffles need every lane
                float mx = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) mx = fmaxf(mx, fmaf(tk, acc[rr][cc], cb[cc] - Lr[rr]));
                mx = max16(mx);
                if (ovf) {
                    const float mn = fmaxf(m[rr], mx);
                    sc[rr] = ex2f(m[rr] - mn);
                    m[rr] = mn;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) w[cc] = ex2f(fmaf(tk, acc[rr][cc], cb[cc] - Lr[rr] - mn));
                }
            }
            if (p.exact_sig) {
                // A pair whose fp32 weight is within 2^-30 / m of a_i is re-evaluated
                // exactly: its exponent, log2 b_j + kappa (f_i + g_j - C_ij), rounds in
                // fp32 at the size of kappa |x||y|, which moves the gradient by ~1e-4 at
                // wide d; the rest carry less than 2^-30 of the row between them.
                const int row = row0 + 4 * tr + rr;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int j = base + 4 * tc + cc;
                    if (row < p.n && j < p.m && fmaf(tk, acc[rr][cc], cb[cc] - Lr[rr]) > sig_thr) {
                        const float e = exact_log2_plan(p.X + (xb + row) * d, p.Yorig + (yb + j) * d, d,
                                                        p.fpot[xb + row], p.gpot[yb + j], 0.f, p.lw2y[yb + j], kap);
                        w[cc] = ex2f(e - m[rr]);
                    }
                }
            }
            float tq = 0.f, trs = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float C = nxr[rr] + nyc[cc] - 2.f * acc[rr][cc];
                tq = fmaf(w[cc], C, tq);
                trs += w[cc];
                Ps[(4 * tr + rr) * (DN_CT + 1) + 4 * tc + cc] = w[cc];
            }
            r_[rr] = r_[rr] * sc[rr] + sum16(trs);
            q_[rr] = q_[rr] * sc[rr] + sum16(tq);
        }
        __syncthreads();
        // the tile's coordinates of this block's slice, if another slice is staged
        if (kb0 + dk < d) {
            dense_stage(Ys, cols, base, DN_CT, p.m, d, kb0, kwz);
            __syncthreads();
        }
        // v[rows][k] += sum_c P[rows][c] * Y[c][kb0 + k], thread owns k = tc + 16 kk
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int kk = 0; kk < KV; ++kk) v[rr][kk] *= sc[rr];
        for (int c = 0; c < DN_CT; ++c) {
            float pv[4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) pv[rr] = Ps[(4 * tr + rr) * (DN_CT + 1) + c];
#pragma unroll
            for (int kk = 0; kk < KV; ++kk) {
                const int k = tc + 16 * kk;
                const float yv = (k < kwz) ? Ys[k * DN_LDT + c] : 0.f;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) v[rr][kk] = fmaf(pv[rr], yv, v[rr][kk]);
            }
        }
    }
    float qsum = 0.f;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int row = row0 + 4 * tr + rr;
        if (row >= p.n) continue;
        const float ai = p.a ? p.a[xb + row] : 1.f / (float)p.n;
        const float fac = ai * ex2f(m[rr]);
        const float ri = r_[rr] * fac;
        if (tc == 0 && blockIdx.z == 0) {
            qsum += q_[rr] * fac;
            if (p.rowsum) p.rowsum[xb + row] = ri;
        }
        if (p.grad) {
            const float* sh = p.shift + (size_t)b * d + kb0;
            const float* xo = p.X + (xb + row) * d + kb0;
            float* gr = p.grad + (xb + row) * d + kb0;
#pragma unroll
            for (int kk = 0; kk < KV; ++kk) {
                const int k = tc + 16 * kk;
                if (k < kwz) gr[k] = 2.f * (ai * xo[k] - fmaf(ri, sh[k], v[rr][kk] * fac));
            }
        }
    }
    if (p.cost_part && blockIdx.z == 0) {
        qsum = block_sum<DN_T>(qsum, red);
        if (threadIdx.x == 0) p.cost_part[b * p.rowtiles + blockIdx.x] = qsum;
    }
}

int dense_apply_rows_per_cta() { return DN_RT; }

cudaError_t launch_dense_apply(const ApplyArgs& p, cudaStream_t st) {
    if (p.d < 1 || p.d > DN_MAXD) return cudaErrorInvalidValue;
    const size_t sm = dense_smem_bytes(p.d) + sizeof(float) * ((size_t)DN_RT * (DN_CT + 1) + DN_CT + 8);
    // above d = 256, one CTA per row block and 256-coordinate slice of the gradient
    dim3 grid(p.rowtiles, p.B, (p.d + DN_DK - 1) / DN_DK), block(DN_T);
    const int kv = (dense_dk(p.d) + 15) / 16;
#define SOT_AP_CASE(KVV)                                                                                   \
    {                                                                                                      \
        cudaError_t e = cudaFuncSetAttribute(dense_apply_kernel<KVV>,                                      \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);        \
        if (e != cudaSuccess) return e;                                                                    \
        count_launches(1); dense_apply_kernel<KVV><<<grid, block, sm, st>>>(p); \
    }
    if (kv <= 1) SOT_AP_CASE(1)
    else if (kv <= 2) SOT_AP_CASE(2)
    else if (kv <= 4) SOT_AP_CASE(4)
    else if (kv <= 8) SOT_AP_CASE(8)
    else SOT_AP_CASE(16)
#undef SOT_AP_CASE
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Thresholded COO, dense.  t_ij = fma(2 kappa, x_i.y_j, log2 b_j - Lam_j) and
// u_ji = fma(2 kappa, x_i.y_j, log2 a_i - L_i) with the dot product
// accumulated k-ascending from zero, exactly as in the maximum pass, so the
// predicate and the maxima agree bit for bit.  One warp per row; lanes take
// 32 consecutive columns; ballot / popc order the writes.  Stored values are
// P_ij with the exponent in float-float (exact_log2_plan).
constexpr int DC_T = 256;
template <bool WRITE>
__global__ void __launch_bounds__(DC_T) dense_coo_kernel(CooArgs p) {
    extern __shared__ float smem[];
    const int d = p.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int i = blockIdx.x * (DC_T / 32) + warp;
    float* xs = smem + warp * d;
    const size_t xb = (size_t)b * p.n, yb = (size_t)b * p.m;
    const bool ok = i < p.n;
    for (int k = lane; k < d; k += 32) xs[k] = ok ? p.xpack[(xb + i) * d + k] : 0.f;
    __syncwarp();
    if (!ok) return;  // whole warp leaves together
    const float thr = p.Mr[xb + i] + p.log2tau;
    const float e_i = p.lw2x[xb + i] - p.L[xb + i];
    const float2 kap = make_float2(p.kap_hi, p.kap_lo);
    long long pos = WRITE ? p.rowptr[xb + i] : 0;
    int cnt = 0;
    for (int base = 0; base < p.m; base += 32) {
        const int j = base + lane;
        bool keep = false;
        float acc = 0.f, c = 0.f;
        if (j < p.m) {
            const float* y = p.ypack + (yb + j) * d;
            for (int k = 0; k < d; ++k) acc = fmaf(xs[k], y[k], acc);
            c = p.lw2y[yb + j] - p.Lam[yb + j];
            if (p.dirs & 1) keep = fmaf(p.two_kappa, acc, c) >= thr;
            if (p.dirs & 2) keep = keep || (fmaf(p.two_kappa, acc, e_i) >= p.Mc[yb + j] + p.log2tau);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, keep);
        if (WRITE) {
            if (keep && pos + __popc(mask & ((1u << lane) - 1u)) < p.capacity) {
                const long long o = pos + __popc(mask & ((1u << lane) - 1u));
                p.rows[o] = i;
                p.cols[o] = j;
                p.vals[o] = exp2f(exact_log2_plan(p.X + (xb + i) * d, p.Y + (yb + j) * d, d, p.f[xb + i],
                                                  p.g[yb + j], p.lw2x[xb + i], p.lw2y[yb + j], kap));
            }
            pos += __popc(mask);
        } else {
            cnt += __popc(mask);
        }
    }
    if (!WRITE && lane == 0) p.counts[xb + i] = cnt;
}

cudaError_t launch_dense_coo(const CooArgs& p, int write_pass, cudaStream_t st) {
    if (p.d < 1 || p.d > DN_MAXD) return cudaErrorInvalidValue;
    dim3 grid((p.n + DC_T / 32 - 1) / (DC_T / 32), p.B), block(DC_T);
    const size_t sm = sizeof(float) * (DC_T / 32) * p.d;
    if (write_pass) { count_launches(1); dense_coo_kernel<true><<<grid, block, sm, st>>>(p); }
    else { count_launches(1); dense_coo_kernel<false><<<grid, block, sm, st>>>(p); }
    return cudaGetLastError();
}

}  // namespace sot
