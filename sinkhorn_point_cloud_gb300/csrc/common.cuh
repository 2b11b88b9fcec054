// common.cuh -- device helpers shared by the sm_103a kernels of libsot.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#define SOT_LN2 0.69314718055994530942f
#define SOT_LOG2E 1.44269504088896340736f

// Hardware base-2 exponential / logarithm (MUFU).  ex2 of -inf is +0; the
// .ftz forms flush subnormal results to zero.
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed two-lane fp32 arithmetic (one instruction, two IEEE results; each
// lane is rounded exactly as the scalar instruction would round it).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\tmov.b64 rc, {%6,%7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0,%1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2,%3};\n\tmov.b64 rb, {%4,%5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0,%1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Error-free transformations: a + b = s + e exactly (Knuth), a * b = p + e
// exactly (FMA); explicitly rounded so the compiler neither fuses nor
// reorders them.
__device__ __forceinline__ float2 two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float z = __fsub_rn(s, a);
    return make_float2(s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z)));
}
__device__ __forceinline__ float2 two_prod(float a, float b) {
    const float q = __fmul_rn(a, b);
    return make_float2(q, __fmaf_rn(a, b, -q));
}

// Float-float (unevaluated hi + lo) arithmetic on top of the error-free
// transformations, renormalised so that |lo| <= ulp(hi) / 2.
__device__ __forceinline__ float2 ff_renorm(float hi, float lo) {
    const float s = __fadd_rn(hi, lo);
    return make_float2(s, __fsub_rn(lo, __fsub_rn(s, hi)));
}
__device__ __forceinline__ float2 ff_add(float2 a, float2 b) {
    const float2 s = two_sum(a.x, b.x);
    return ff_renorm(s.x, __fadd_rn(s.y, __fadd_rn(a.y, b.y)));
}
__device__ __forceinline__ float2 ff_mul(float2 a, float2 b) {
    const float2 q = two_prod(a.x, b.x);
    return ff_renorm(q.x, __fmaf_rn(a.x, b.y, __fmaf_rn(a.y, b.x, q.y)));
}

// log2 P_ij = log2 w_i + log2 w'_j + kappa (f_i + g_j - C_ij) in float-float:
// C_ij from error-free coordinate differences and squares of the caller's
// points, the potentials and C_ij cancelling exactly before the product with
// kappa = kap.x + kap.y.  Accurate to a few fp32 ulps of the (small) result,
// where fp32 would round at the size of kappa |f_i|.
__device__ __forceinline__ float exact_log2_plan(const float* x, const float* y, int d, float fi, float gj,
                                                 float lwi, float lwj, float2 kap) {
    float2 C2 = make_float2(0.f, 0.f);
    for (int k = 0; k < d; ++k) {
        const float2 dd = two_sum(x[k], -y[k]);
        float2 sq = two_prod(dd.x, dd.x);
        sq.y = __fmaf_rn(2.f * dd.x, dd.y, sq.y);
        C2 = ff_add(C2, sq);
    }
    const float2 pot = ff_add(two_sum(fi, gj), make_float2(-C2.x, -C2.y));
    const float2 ell = ff_add(ff_mul(kap, pot), two_sum(lwi, lwj));
    return __fadd_rn(ell.x, ell.y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide reductions (fixed tree => deterministic).  `red` must hold one
// float per warp.  Every thread of the block must call them.
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x < 32) {
        t = (l < NT / 32) ? red[l] : 0.f;
        t = warp_sum(t);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}
template <int NT>
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = -INFINITY;
    if (threadIdx.x < 32) {
        t = (l < NT / 32) ? red[l] : -INFINITY;
        t = warp_max(t);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

// Row-state stabiliser handling shared by the half-step kernels.
// A row's running log2-sum is (m, s): value = m + log2(s).
// The tile sum is considered unsafe (overflow risk) above this bound.
#define SOT_TILE_SUM_MAX 1.2676506e30f  /* 2^100 */
// Below this bound the final sum may have lost precision to flushed terms.
#define SOT_SUM_MIN 8.2718061e-25f      /* 2^-80 */
// The warm stabiliser sits this many log2 units below the previous row value.
#define SOT_STAB_BIAS 32.0f

// Combine two (m, s) partial log2-sums.
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY || s2 == 0.f) return;
    if (m == -INFINITY || s == 0.f) { m = m2; s = s2; return; }
    if (m2 > m) { s = s * ex2f(m - m2) + s2; m = m2; }
    else        { s = s + s2 * ex2f(m2 - m); }
}

// Order-preserving float <-> unsigned map (for atomicMin on floats):
// unsigned order of the keys equals the numeric order of the floats.
#define SOT_ORD_EMPTY 0xFFFFFFFFu  /* identity of the minimum */
__device__ __forceinline__ unsigned ord_encode(float v) {
    const unsigned u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_decode(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Stabiliser of a row at the start of a half-step.  With a per-cloud bound
// lo = min over the other side of (state_before - state_after) from the
// half-step that produced the current column state, the new row value
// satisfies L_new >= L_old + lo, so starting at m = L_old + lo keeps the row
// sum >= 1 (no underflow).  Without a bound: previous value minus a bias,
// or -inf on a cold start.
__device__ __forceinline__ float stabiliser(int cold, const unsigned* lo_in, int b, float old) {
    if (cold) return -INFINITY;
    if (lo_in) {
        const float lo = ord_decode(lo_in[b]);
        if (isfinite(lo)) return old + lo;
    }
    return old - SOT_STAB_BIAS;
}

// Device status bits (OR-ed into a status word).
#define SOT_DEV_RETRY_ROWS 1  /* some rows took the slow full-row recompute */
#define SOT_DEV_BAD_COO 2     /* COO input unsorted / out of range */
#define SOT_DEV_TIMEOUT 4     /* a bounded device-side wait gave up */
