// k_point.cu -- fused Sinkhorn half-steps for point clouds with d <= 3 on
// FP32 FMA + MUFU ex2 (no tensor cores: a 3-term distance is no dense
// contraction).
//
// One half-step ("FlashSinkhorn", Methodologie 1-2) for row i of the updated
// side, in base 2 with kappa = 1/(eps ln 2) and the state L_i = -kappa f_i
// (Lam_j = -kappa g_j):
//     L_i = log2 sum_j 2^( c_j - kappa |x_i - y_j|^2 ),   c_j = log2 w_j - Lam_j
// The squared distance is formed in the direct form from coordinates scaled
// by sqrt(kappa): in fp32 the expanded form 2 kappa x.y - kappa |y|^2 rounds at
// the magnitude of kappa |x||y| and, at eps = 1e-2 on unit-sphere clouds, moved
// the gradient by ~1e-4 relative; the direct form rounds at the magnitude of
// the (small) distances that matter and stays near 5e-6.
// The score tile is formed in registers from a column tile staged in shared
// memory and never stored; the row-wise log-sum-exp is accumulated on chip
// (Methodologie 2, "Online LSE"), one row block stays resident while every
// column tile streams past it (row-stationary traversal).
//
// Stabiliser.  Each row keeps a running (m, s) with value m + log2 s; m starts
// at a bound that keeps the sum >= 1 (see stabiliser() in common.cuh) or -inf
// on a cold start, so a column costs 3 FADD + 3 FFMA + 1 FADD + 1 ex2 + 1 FADD
// and no per-pair max.  A tile whose sum leaves the safe range is recomputed
// against the tile maximum, so the result is the exact LSE for any start.
//
// Layout of a column tile in shared memory: column pairs interleaved so that
// one 16-byte load yields two 2-lane operands of the packed f32x2 arithmetic:
//     tile[2p]   = (-v_j.x, -v_j'.x, -v_j.y, -v_j'.y),
//     tile[2p+1] = (-v_j.z, -v_j'.z, -c_j,   -c_j')      with v = sqrt(kappa) y.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace sot {

constexpr int PT_T = 128;               // threads per CTA
constexpr int PT_TC = 2 * PT_T;         // columns per shared-memory tile
// Rows per thread (RPT) is 4, 2 or 1: a CTA holds PT_T * RPT rows.  More rows
// per thread reuse each staged column for more rows; fewer give more row
// blocks, so that a workload of few, short rows still fills the GPU with CTAs
// that each cover several column tiles (see point_plan).

int point_cols_per_tile() { return PT_TC; }

// Score relative to a base: acc = base + |u - v|^2 with d = u + (-v), fp32 in
// this fixed order (the maximum passes and the COO predicate evaluate the same
// chain, so their decisions agree bit for bit).  The score is t = m - acc when
// base = m - c.
template <int D>
__device__ __forceinline__ float2 pair_chain(float2 acc, float2 u0, float2 u1, float2 u2, float4 A, float4 Bv) {
    if (D >= 1) { const float2 d = fadd2(u0, make_float2(A.x, A.y)); acc = ffma2(d, d, acc); }
    if (D >= 2) { const float2 d = fadd2(u1, make_float2(A.z, A.w)); acc = ffma2(d, d, acc); }
    if (D >= 3) { const float2 d = fadd2(u2, make_float2(Bv.x, Bv.y)); acc = ffma2(d, d, acc); }
    return acc;
}
// Scalar form of the same chain for one (row, column): u = scaled row point,
// nv = negated scaled column point, base = m - c.  Written with explicitly
// rounded intrinsics so the compiler can neither contract nor pair these
// operations: the maximum pass and both COO passes must produce the same bits.
template <int D>
__device__ __forceinline__ float scalar_chain(float base, float u0, float u1, float u2, float nv0, float nv1,
                                              float nv2) {
    float acc = base;
    if (D >= 1) { const float d = __fadd_rn(u0, nv0); acc = __fmaf_rn(d, d, acc); }
    if (D >= 2) { const float d = __fadd_rn(u1, nv1); acc = __fmaf_rn(d, d, acc); }
    if (D >= 3) { const float d = __fadd_rn(u2, nv2); acc = __fmaf_rn(d, d, acc); }
    return acc;
}
// Scaled point and negated column bias, computed the same way everywhere.
__device__ __forceinline__ float scaled(float sk, float v) { return __fmul_rn(sk, v); }
__device__ __forceinline__ float neg_bias(float w2, float state) { return -__fsub_rn(w2, state); }

// Stage columns [base, base + PT_TC) of the chunk ending at c_end: scaled,
// negated coordinates and the negated column bias.
__device__ __forceinline__ void load_point_tile(float4* tile, const float4* cp, const float* cst, int base,
                                                int c_end, float sk) {
    const int j0 = base + 2 * threadIdx.x, j1 = j0 + 1;
    float4 c0 = make_float4(0.f, 0.f, 0.f, INFINITY), c1 = c0;  // padding: -c = +inf -> score -inf
    if (j0 < c_end) {
        const float4 y = cp[j0];
        c0 = make_float4(-scaled(sk, y.x), -scaled(sk, y.y), -scaled(sk, y.z), neg_bias(y.w, cst[j0]));
    }
    if (j1 < c_end) {
        const float4 y = cp[j1];
        c1 = make_float4(-scaled(sk, y.x), -scaled(sk, y.y), -scaled(sk, y.z), neg_bias(y.w, cst[j1]));
    }
    tile[2 * threadIdx.x] = make_float4(c0.x, c1.x, c0.y, c1.y);
    tile[2 * threadIdx.x + 1] = make_float4(c0.z, c1.z, c0.w, c1.w);
}

// Two-pass LSE of one full row by the whole CTA (slow path for rows whose
// stabilised sum underflowed).  Returns log2 sum_j 2^(score_j).
template <int D>
__device__ float point_row_full(const float4* cp, const float* cst, int nc, float u0, float u1, float u2, float sk,
                                float* red) {
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < nc; j += PT_T) {
        const float4 c = cp[j];
        mx = fmaxf(mx, -scalar_chain<D>(-(c.w - cst[j]), u0, u1, u2, -(sk * c.x), -(sk * c.y), -(sk * c.z)));
    }
    mx = block_max<PT_T>(mx, red);
    if (mx == -INFINITY) return -INFINITY;
    float sm = 0.f;
    for (int j = threadIdx.x; j < nc; j += PT_T) {
        const float4 c = cp[j];
        sm += ex2f(-scalar_chain<D>(-(c.w - cst[j]), u0, u1, u2, -(sk * c.x), -(sk * c.y), -(sk * c.z)) - mx);
    }
    sm = block_sum<PT_T>(sm, red);
    return mx + log2f(sm);
}

template <int D, int MODE, int PT_RPT>
__global__ void __launch_bounds__(PT_T) point_half_kernel(HalfArgs p) {
    constexpr int PT_ROWS = PT_T * PT_RPT;  // rows per CTA
    if (p.stop_flag && *(volatile const int*)p.stop_flag) return;
    __shared__ float4 tile[PT_TC];
    __shared__ float red[PT_T / 32];
    __shared__ int s_last;
    __shared__ int s_nretry;
    __shared__ int s_retry[PT_ROWS];

    const int b = blockIdx.y;
    const int rt = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rt * PT_ROWS;
    const int c_begin = ch * p.chunk;
    const int c_end = min(p.nc, c_begin + p.chunk);
    const float4* rp = reinterpret_cast<const float4*>(p.rpack) + (size_t)b * p.nr;
    const float4* cp = reinterpret_cast<const float4*>(p.cpack) + (size_t)b * p.nc;
    const float* cst = p.cstate + (size_t)b * p.nc;
    const size_t rbase = (size_t)b * p.nr;

    if (p.lo_reset && blockIdx.x == 0 && blockIdx.y == 0)
        for (int k = threadIdx.x; k < p.B; k += PT_T) p.lo_reset[k] = SOT_ORD_EMPTY;
    const float sk = sqrtf(0.5f * p.two_kappa);  // sqrt(kappa)
    float2 q0[PT_RPT], q1[PT_RPT], q2[PT_RPT], nm[PT_RPT];
    float m[PT_RPT], s[PT_RPT], old[PT_RPT];
#pragma unroll
    for (int r = 0; r < PT_RPT; ++r) {
        const int row = row0 + threadIdx.x + r * PT_T;
        const bool valid = row < p.nr;
        float4 x = valid ? rp[row] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float a0 = scaled(sk, x.x), a1 = scaled(sk, x.y), a2 = scaled(sk, x.z);  // scaled row point u
        q0[r] = make_float2(a0, a0);
        q1[r] = make_float2(a1, a1);
        q2[r] = make_float2(a2, a2);
        old[r] = (MODE == MODE_LSE && valid && p.rstate_in) ? p.rstate_in[rbase + row] : 0.f;
        if (MODE == MODE_MAX) {
            m[r] = -INFINITY;
        } else if (!valid) {
            m[r] = INFINITY;  // every term becomes 2^-inf = 0; never written
        } else {
            m[r] = stabiliser(p.cold, p.lo_in, b, old[r]);
        }
        nm[r] = make_float2(m[r], m[r]);  // base of the chain: m - c
        s[r] = 0.f;
    }

    for (int base = c_begin; base < c_end; base += PT_TC) {
        __syncthreads();
        load_point_tile(tile, cp, cst, base, c_end, sk);
        __syncthreads();
        if (MODE == MODE_MAX) {
            float2 mx[PT_RPT];
#pragma unroll
            for (int r = 0; r < PT_RPT; ++r) mx[r] = make_float2(-INFINITY, -INFINITY);
#pragma unroll 4
            for (int pp = 0; pp < PT_TC / 2; ++pp) {
                const float4 A = tile[2 * pp], Bv = tile[2 * pp + 1];
#pragma unroll
                for (int r = 0; r < PT_RPT; ++r) {
                    // scalar chain: the COO predicate re-evaluates exactly these bits
                    const float a0 = scalar_chain<D>(Bv.z, q0[r].x, q1[r].x, q2[r].x, A.x, A.z, Bv.x);
                    const float a1 = scalar_chain<D>(Bv.w, q0[r].x, q1[r].x, q2[r].x, A.y, A.w, Bv.y);
                    mx[r].x = fmaxf(mx[r].x, -a0);
                    mx[r].y = fmaxf(mx[r].y, -a1);
                }
            }
#pragma unroll
            for (int r = 0; r < PT_RPT; ++r) m[r] = fmaxf(m[r], fmaxf(mx[r].x, mx[r].y));
        } else {
            float2 st[PT_RPT];
#pragma unroll
            for (int r = 0; r < PT_RPT; ++r) st[r] = make_float2(0.f, 0.f);
#pragma unroll 4
            for (int pp = 0; pp < PT_TC / 2; ++pp) {
                const float4 A = tile[2 * pp], Bv = tile[2 * pp + 1];
                const float2 ncj = make_float2(Bv.z, Bv.w);
#pragma unroll
                for (int r = 0; r < PT_RPT; ++r) {
                    const float2 acc = pair_chain<D>(fadd2(nm[r], ncj), q0[r], q1[r], q2[r], A, Bv);  // m - t
                    st[r] = fadd2(st[r], make_float2(ex2f(-acc.x), ex2f(-acc.y)));
                }
            }
#pragma unroll
            for (int r = 0; r < PT_RPT; ++r) {
                float ts = st[r].x + st[r].y;
                if (!(ts < SOT_TILE_SUM_MAX)) {
                    // slow path: re-stabilise this row on the tile maximum
                    float mt = -INFINITY;
                    for (int pp = 0; pp < PT_TC / 2; ++pp) {
                        const float4 A = tile[2 * pp], Bv = tile[2 * pp + 1];
                        const float2 acc = pair_chain<D>(make_float2(Bv.z, Bv.w), q0[r], q1[r], q2[r], A, Bv);
                        mt = fmaxf(mt, fmaxf(-acc.x, -acc.y));
                    }
                    const float mn = fmaxf(m[r], mt);
                    if (mn == -INFINITY) {
                        ts = 0.f;
                    } else {
                        s[r] = (m[r] == -INFINITY) ? 0.f : s[r] * ex2f(m[r] - mn);
                        m[r] = mn;
                        nm[r] = make_float2(mn, mn);
                        float2 sum = make_float2(0.f, 0.f);
                        for (int pp = 0; pp < PT_TC / 2; ++pp) {
                            const float4 A = tile[2 * pp], Bv = tile[2 * pp + 1];
                            const float2 acc = pair_chain<D>(fadd2(nm[r], make_float2(Bv.z, Bv.w)), q0[r], q1[r],
                                                             q2[r], A, Bv);
                            sum = fadd2(sum, make_float2(ex2f(-acc.x), ex2f(-acc.y)));
                        }
                        ts = sum.x + sum.y;
                    }
                }
                s[r] += ts;
            }
        }
    }

    // ---- combine column chunks -------------------------------------------
    if (p.split > 1) {
        const size_t stride = (size_t)p.B * p.nr;
#pragma unroll
        for (int r = 0; r < PT_RPT; ++r) {
            const int row = row0 + threadIdx.x + r * PT_T;
            if (row < p.nr) {
                p.part_m[ch * stride + rbase + row] = m[r];
                if (MODE == MODE_LSE) p.part_s[ch * stride + rbase + row] = s[r];
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned prev = atomicAdd(&p.counters[b * p.rowtiles + rt], 1u);
            s_last = (prev == (unsigned)(p.split - 1));
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
#pragma unroll
        for (int r = 0; r < PT_RPT; ++r) {
            const int row = row0 + threadIdx.x + r * PT_T;
            if (row >= p.nr) continue;
            float M = -INFINITY, S = 0.f;
            for (int c = 0; c < p.split; ++c) {
                const float pm = __ldcg(p.part_m + c * stride + rbase + row);
                if (MODE == MODE_MAX) {
                    M = fmaxf(M, pm);
                } else {
                    lse_combine(M, S, pm, __ldcg(p.part_s + c * stride + rbase + row));
                }
            }
            m[r] = M;
            s[r] = S;
        }
        if (threadIdx.x == 0) p.counters[b * p.rowtiles + rt] = 0u;
    }

    // ---- finalise rows ----------------------------------------------------
    if (threadIdx.x == 0) s_nretry = 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < PT_RPT; ++r) {
        const int row = row0 + threadIdx.x + r * PT_T;
        if (row >= p.nr) continue;
        if (MODE == MODE_MAX) {
            p.rstate_out[rbase + row] = m[r];
        } else if (s[r] >= SOT_SUM_MIN && s[r] < INFINITY && m[r] > -INFINITY) {
            p.rstate_out[rbase + row] = m[r] + log2f(s[r]);
        } else {
            s_retry[atomicAdd(&s_nretry, 1)] = row;
        }
    }
    __syncthreads();
    if (MODE == MODE_LSE) {
        const int nretry = s_nretry;
        for (int k = 0; k < nretry; ++k) {
            const int row = s_retry[k];
            const float4 x = rp[row];
            const float v = point_row_full<D>(cp, cst, p.nc, sk * x.x, sk * x.y, sk * x.z, sk, red);
            if (threadIdx.x == 0) {
                p.rstate_out[rbase + row] = v;
                atomicOr(p.status, SOT_DEV_RETRY_ROWS);
            }
        }
        if (p.errpart || p.lo_out) {
            __syncthreads();
            float e = 0.f, lo = INFINITY;
            const float wu = 1.f / (float)p.nr;
#pragma unroll
            for (int r = 0; r < PT_RPT; ++r) {
                const int row = row0 + threadIdx.x + r * PT_T;
                if (row >= p.nr) continue;
                const float nv = p.rstate_out[rbase + row];
                const float w = p.rweight ? p.rweight[rbase + row] : wu;
                e += w * fabsf(ex2f(nv - old[r]) - 1.f);
                lo = fminf(lo, old[r] - nv);
            }
            if (p.errpart) {
                e = block_sum<PT_T>(e, red);
                if (threadIdx.x == 0) p.errpart[b * p.rowtiles + rt] = e;
            }
            if (p.lo_out) {
                lo = warp_min(lo);
                if ((threadIdx.x & 31) == 0 && lo < INFINITY) atomicMin(p.lo_out + b, ord_encode(lo));
            }
        }
    }
}

using PointKernel = void (*)(HalfArgs);

template <int RPT>
static PointKernel point_kernel_rpt(int d, int mode) {
    const bool mx = mode == MODE_MAX;
    switch (d) {
        case 1: return mx ? point_half_kernel<1, MODE_MAX, RPT> : point_half_kernel<1, MODE_LSE, RPT>;
        case 2: return mx ? point_half_kernel<2, MODE_MAX, RPT> : point_half_kernel<2, MODE_LSE, RPT>;
        case 3: return mx ? point_half_kernel<3, MODE_MAX, RPT> : point_half_kernel<3, MODE_LSE, RPT>;
        default: return nullptr;
    }
}

static PointKernel point_kernel(int d, int mode, int rpt) {
    return rpt == 1 ? point_kernel_rpt<1>(d, mode) : rpt == 2 ? point_kernel_rpt<2>(d, mode) : rpt == 4 ? point_kernel_rpt<4>(d, mode) : nullptr;
}

cudaError_t launch_point_half(const HalfArgs& p, int mode, cudaStream_t st) {
    const PointKernel k = point_kernel(p.d, mode, p.rpt);
    if (!k || p.rowtiles != (p.nr + PT_T * p.rpt - 1) / (PT_T * p.rpt)) return cudaErrorInvalidValue;
    dim3 grid(p.rowtiles * p.split, p.B), block(PT_T);
    count_launches(1);
    k<<<grid, block, 0, st>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Plan application ("FlashSinkhorn", Methodologie 3): per row, with the given
// potentials and P_ij / a_i = 2^(kappa nx_i - L_i + kappa ny_j + log2 b_j - Lam_j - kappa C_ij),
//   r_i = sum_j P_ij,  v_i = sum_j P_ij y_j,  q_i = sum_j P_ij C_ij
// with C_ij in the direct form |x_i - y_j|^2 (accurate for near-coincident
// points).  Outputs cost = sum_i q_i (per-CTA partials), grad_i =
// 2 (a_i x_i - sum_j P_ij y_j) in the caller's coordinates, rowsum r_i.
constexpr int AP_T = 128;
constexpr int AP_TC = 256;
int point_apply_rows_per_cta() { return AP_T; }

template <int D>
__global__ void __launch_bounds__(AP_T) point_apply_kernel(ApplyArgs p) {
    __shared__ float4 tile[AP_TC];
    __shared__ float red[AP_T / 32];
    const int b = blockIdx.y;
    const int row = blockIdx.x * AP_T + threadIdx.x;
    const bool valid = row < p.n;
    const float4* xp = reinterpret_cast<const float4*>(p.xpack) + (size_t)b * p.n;
    const float4* yp = reinterpret_cast<const float4*>(p.ypack) + (size_t)b * p.m;
    const float* ny = p.ny + (size_t)b * p.m;
    const float* lam = p.Lam + (size_t)b * p.m;
    const float4 x = valid ? xp[row] : make_float4(0.f, 0.f, 0.f, 0.f);
    // row part of the exponent, relative to the row weight
    const float A = valid ? p.kappa * p.nx[(size_t)b * p.n + row] - p.L[(size_t)b * p.n + row] : 0.f;
    float m = valid ? -SOT_STAB_BIAS : INFINITY;
    float r = 0.f, v0 = 0.f, v1 = 0.f, v2 = 0.f, q = 0.f;
    for (int base = 0; base < p.m; base += AP_TC) {
        __syncthreads();
        for (int t = threadIdx.x; t < AP_TC; t += AP_T) {
            const int j = base + t;
            float4 c = make_float4(0.f, 0.f, 0.f, -INFINITY);
            if (j < p.m) {
                c = yp[j];
                c.w = fmaf(p.kappa, ny[j], c.w - lam[j]);
            }
            tile[t] = c;
        }
        __syncthreads();
        const float Am = A - m;
        float tr = 0.f, t0 = 0.f, t1 = 0.f, t2 = 0.f, tq = 0.f;
#pragma unroll 4
        for (int t = 0; t < AP_TC; ++t) {
            const float4 c = tile[t];
            const float d0 = x.x - c.x, d1 = x.y - c.y, d2 = x.z - c.z;
            float C = d0 * d0;
            if (D >= 2) C = fmaf(d1, d1, C);
            if (D >= 3) C = fmaf(d2, d2, C);
            const float w = ex2f(fmaf(-p.kappa, C, Am + c.w));
            tr += w;
            t0 = fmaf(w, c.x, t0);
            if (D >= 2) t1 = fmaf(w, c.y, t1);
            if (D >= 3) t2 = fmaf(w, c.z, t2);
            tq = fmaf(w, C, tq);
        }
        if (!(tr < SOT_TILE_SUM_MAX)) {
            float mt = -INFINITY;
            for (int t = 0; t < AP_TC; ++t) {
                const float4 c = tile[t];
                const float d0 = x.x - c.x, d1 = x.y - c.y, d2 = x.z - c.z;
                float C = d0 * d0;
                if (D >= 2) C = fmaf(d1, d1, C);
                if (D >= 3) C = fmaf(d2, d2, C);
                mt = fmaxf(mt, fmaf(-p.kappa, C, A + c.w));
            }
            const float mn = fmaxf(m, mt);
            const float sc = ex2f(m - mn);
            r *= sc; v0 *= sc; v1 *= sc; v2 *= sc; q *= sc;
            m = mn;
            const float Am2 = A - m;
            tr = t0 = t1 = t2 = tq = 0.f;
            for (int t = 0; t < AP_TC; ++t) {
                const float4 c = tile[t];
                const float d0 = x.x - c.x, d1 = x.y - c.y, d2 = x.z - c.z;
                float C = d0 * d0;
                if (D >= 2) C = fmaf(d1, d1, C);
                if (D >= 3) C = fmaf(d2, d2, C);
                const float w = ex2f(fmaf(-p.kappa, C, Am2 + c.w));
                tr += w;
                t0 = fmaf(w, c.x, t0);
                if (D >= 2) t1 = fmaf(w, c.y, t1);
                if (D >= 3) t2 = fmaf(w, c.z, t2);
                tq = fmaf(w, C, tq);
            }
        }
        r += tr; v0 += t0; v1 += t1; v2 += t2; q += tq;
    }
    float qi = 0.f;
    if (valid) {
        const float ai = p.a ? p.a[(size_t)b * p.n + row] : 1.f / (float)p.n;
        const float fac = ai * ex2f(m);
        r *= fac; v0 *= fac; v1 *= fac; v2 *= fac; qi = q * fac;
        if (p.rowsum) p.rowsum[(size_t)b * p.n + row] = r;
        if (p.grad) {
            // v_i in caller coordinates: sum_j P_ij (y'_j + t) = v'_i + r_i t
            const float* sh = p.shift + (size_t)b * D;
            const float* xo = p.X + ((size_t)b * p.n + row) * D;
            float* gr = p.grad + ((size_t)b * p.n + row) * D;
            const float vv[3] = {v0, v1, v2};
#pragma unroll
            for (int k = 0; k < D; ++k) gr[k] = 2.f * (ai * xo[k] - fmaf(r, sh[k], vv[k]));
        }
    }
    if (p.cost_part) {
        qi = block_sum<AP_T>(qi, red);
        if (threadIdx.x == 0) p.cost_part[b * p.rowtiles + blockIdx.x] = qi;
    }
}

cudaError_t launch_point_apply(const ApplyArgs& p, cudaStream_t st) {
    dim3 grid(p.rowtiles, p.B), block(AP_T);
    switch (p.d) {
        case 1: count_launches(1); point_apply_kernel<1><<<grid, block, 0, st>>>(p); break;
        case 2: count_launches(1); point_apply_kernel<2><<<grid, block, 0, st>>>(p); break;
        case 3: count_launches(1); point_apply_kernel<3><<<grid, block, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Thresholded COO plan ("CUDA-Optimized APML", Abstract / Innovation).
// Pair (i, j) is kept when
//   (dirs & 1) and t_ij >= Mr_i + log2 tau   (row-relative), or
//   (dirs & 2) and u_ji >= Mc_j + log2 tau   (column-relative),
// with t_ij = c_j - kappa|x_i - y_j|^2 (c_j = log2 b_j - Lam_j) and
// u_ji = e_i - kappa|x_i - y_j|^2 (e_i = log2 a_i - L_i), each evaluated by the
// same fp32 chain as the maximum pass of its half (the scaled difference
// u - v is exactly the negation of v - u, so both directions see the same
// squares); the maxima and the predicate therefore agree bit for bit.  A kept
// pair stores P_ij = 2^(log2 a_i + log2 b_j + kappa (f_i + g_j - C_ij)) with
// the exponent in float-float from the caller's points and potentials
// (exact_log2_plan), so the value does not carry the fp32 rounding of the
// large, cancelling terms kappa f_i and kappa g_j.  One
// warp owns CO_RW rows; its lanes take 32 consecutive columns, and a ballot /
// popc over the predicate gives each kept pair its slot, so a row's entries
// come out in ascending column order with coalesced stores.
constexpr int CO_T = 256;
constexpr int CO_RW = 4;                      // rows per warp
constexpr int CO_ROWS = (CO_T / 32) * CO_RW;  // rows per CTA
constexpr int CO_TC = 256;                    // columns per tile

template <int D, bool WRITE>
__global__ void __launch_bounds__(CO_T) point_coo_kernel(CooArgs p) {
    __shared__ float cy[CO_TC];    // -c_j  with c_j = log2 b_j - Lam_j
    __shared__ float4 cv[CO_TC];   // (-sqrt(kappa) y, Mc_j + log2 tau)
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rowb = blockIdx.x * CO_ROWS + warp * CO_RW;
    const float4* xp = reinterpret_cast<const float4*>(p.xpack) + (size_t)b * p.n;
    const float4* yp = reinterpret_cast<const float4*>(p.ypack) + (size_t)b * p.m;
    const size_t xb = (size_t)b * p.n, yb = (size_t)b * p.m;
    const float sk = sqrtf(p.kappa);
    const float2 kap = make_float2(p.kap_hi, p.kap_lo);

    float4 x[CO_RW];
    float u0[CO_RW], u1[CO_RW], u2[CO_RW], thr_r[CO_RW], ne_r[CO_RW];
    long long pos[CO_RW];
    int cnt[CO_RW];
#pragma unroll
    for (int r = 0; r < CO_RW; ++r) {
        const int i = rowb + r;
        const bool ok = i < p.n;
        x[r] = ok ? xp[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        u0[r] = scaled(sk, x[r].x);
        u1[r] = scaled(sk, x[r].y);
        u2[r] = scaled(sk, x[r].z);
        thr_r[r] = ok ? __fadd_rn(p.Mr[xb + i], p.log2tau) : INFINITY;
        ne_r[r] = ok ? neg_bias(x[r].w, p.L[xb + i]) : 0.f;  // -(log2 a_i - L_i)
        pos[r] = (WRITE && ok) ? p.rowptr[xb + i] : 0;
        cnt[r] = 0;
    }
    for (int base = 0; base < p.m; base += CO_TC) {
        __syncthreads();
        for (int t = threadIdx.x; t < CO_TC; t += CO_T) {
            const int j = base + t;
            float c = INFINITY;
            float4 c2 = make_float4(0.f, 0.f, 0.f, INFINITY);
            if (j < p.m) {
                const float4 y = yp[j];
                c = neg_bias(y.w, p.Lam[yb + j]);
                c2 = make_float4(-scaled(sk, y.x), -scaled(sk, y.y), -scaled(sk, y.z),
                                 __fadd_rn(p.Mc[yb + j], p.log2tau));
            }
            cy[t] = c;
            cv[t] = c2;
        }
        __syncthreads();
        for (int cc = 0; cc < CO_TC; cc += 32) {
            const int t = cc + lane;
            const int j = base + t;
            const float c = cy[t];
            const float4 c2 = cv[t];
#pragma unroll
            for (int r = 0; r < CO_RW; ++r) {
                bool keep = false;
                const float trow = -scalar_chain<D>(c, u0[r], u1[r], u2[r], c2.x, c2.y, c2.z);
                if (p.dirs & 1) keep = trow >= thr_r[r];
                if (p.dirs & 2) {
                    // column direction: rows Y, columns X; d = v + (-u) = -(u - v) exactly
                    const float ucol = -scalar_chain<D>(ne_r[r], -c2.x, -c2.y, -c2.z, -u0[r], -u1[r], -u2[r]);
                    keep = keep || (ucol >= c2.w);
                }
                keep = keep && (j < p.m) && (rowb + r < p.n);
                const unsigned mask = __ballot_sync(0xffffffffu, keep);
                if (WRITE) {
                    const long long o = pos[r] + __popc(mask & ((1u << lane) - 1u));
                    if (keep && o < p.capacity) {
                        const int i = rowb + r;
                        const float l2 = exact_log2_plan(p.X + (xb + i) * D, p.Y + (yb + j) * D, D, p.f[xb + i],
                                                         p.g[yb + j], x[r].w, yp[j].w, kap);
                        p.rows[o] = i;
                        p.cols[o] = j;
                        p.vals[o] = exp2f(l2);
                    }
                    pos[r] += __popc(mask);
                } else {
                    cnt[r] += __popc(mask);
                }
            }
        }
    }
    if (!WRITE && lane == 0) {
#pragma unroll
        for (int r = 0; r < CO_RW; ++r)
            if (rowb + r < p.n) p.counts[xb + rowb + r] = cnt[r];
    }
}

cudaError_t launch_point_coo(const CooArgs& p, int write_pass, cudaStream_t st) {
    dim3 grid((p.n + CO_ROWS - 1) / CO_ROWS, p.B), block(CO_T);
#define SOT_CO_CASE(DD)                                                           \
    case DD:                                                                      \
        if (write_pass) { count_launches(1); point_coo_kernel<DD, true><<<grid, block, 0, st>>>(p); } \
        else { count_launches(1); point_coo_kernel<DD, false><<<grid, block, 0, st>>>(p); } \
        break;
    switch (p.d) {
        SOT_CO_CASE(1)
        SOT_CO_CASE(2)
        SOT_CO_CASE(3)
        default: return cudaErrorInvalidValue;
    }
#undef SOT_CO_CASE
    return cudaGetLastError();
}

// Resident CTAs per SM of the half-step kernel with `rpt` rows per thread.
// Cached after the first successful query (the kernel's resources do not
// depend on the device); a failed query returns 4 and is not cached.
static int point_blocks_per_sm(int rpt) {
    static std::atomic<int> occ[3] = {};
    const int slot = rpt == 1 ? 0 : rpt == 2 ? 1 : 2;
    int v = occ[slot].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, point_kernel(3, MODE_LSE, rpt), PT_T, 0) != cudaSuccess ||
        v < 1) {
        cudaGetLastError();
        return 4;
    }
    occ[slot].store(v, std::memory_order_relaxed);
    return v;
}

// Rows per thread and column split of a half-step over B clouds of nr rows
// and nc columns.  For each choice of rows per thread r the split is the one
// of fewest rounds of CTAs per unit of work (a 1 % charge per extra chunk for
// the combining step); the choices are then compared by the work each SM
// carries: its CTAs times r * (column tiles * PT_PAIR[r] + PT_FIXED), where
// PT_PAIR is the cost of a pair relative to 4 rows per thread (each staged
// column feeds fewer rows) and PT_FIXED the per-row work that does not depend
// on the chunk's length (loading and stabilising the rows, combining the
// chunks, finishing the rows), in tiles.  Both were fitted to the half-step
// times of the three d = 3 workloads of 65536 rows (2048, 8192 and 16384
// columns) with 4, 2 and 1 rows per thread.  An SM holding fewer than 16 warps
// is charged for the lanes they leave idle.
constexpr double PT_FIXED = 0.2;

static double pt_pair_cost(int r) { return r == 4 ? 1.0 : r == 2 ? 1.06 : 1.12; }

void point_plan(int B, int nr, int nc, int sms, int* rpt, int* split, int* chunk, int* rowtiles) {
    const int ntiles = (nc + PT_TC - 1) / PT_TC;
    const int smax = ntiles < 64 ? ntiles : 64;
    const long long nsm = sms > 0 ? sms : 1;
    double best_cost = 1e300;
    int br = 4, bs = 1;
    for (int r = 4; r >= 1; r /= 2) {
        const long long base = (long long)B * ((nr + PT_T * r - 1) / (PT_T * r));
        const long long occ = point_blocks_per_sm(r);
        const long long slots = nsm * occ;
        double best = 1e300;
        int s_r = 1;
        for (int s = 1; s <= smax; ++s) {
            const long long units = base * s;
            const double rounds = (double)((units + slots - 1) / slots);
            const double t = rounds / s * (1.0 + 0.01 * (s - 1));
            if (t < best * 0.999) {
                best = t;
                s_r = s;
            }
        }
        const int tpc = (ntiles + s_r - 1) / s_r;
        const long long units = base * ((ntiles + tpc - 1) / tpc);
        const long long per_sm = (units + nsm - 1) / nsm;
        const long long resident = per_sm < occ ? per_sm : occ;
        const double starve = resident * 4 < 16 ? 16.0 / (double)(resident * 4) : 1.0;
        const double cost = (double)per_sm * r * (tpc * pt_pair_cost(r) + PT_FIXED) * starve;
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            br = r;
            bs = s_r;
        }
    }
    *rpt = br;
    *rowtiles = (nr + PT_T * br - 1) / (PT_T * br);
    const int tiles_per_chunk = (ntiles + bs - 1) / bs;
    *chunk = tiles_per_chunk * PT_TC;
    *split = (nc + *chunk - 1) / *chunk;
}

}  // namespace sot
