// k_cluster.cu -- cluster-resident Sinkhorn iterations for small point clouds
// (d <= 3, both clouds together a few thousand points).
//
// The streaming half-step kernels (k_point.cu) pay a launch, a pass over
// global memory for the states and a cross-CTA merge per half-step.  For a
// cloud pair that fits in shared memory that fixed cost dominates: 65536
// pairs of the 256-point workload take 14 us per half-step, almost all of it
// overhead.  Here one thread-block cluster per cloud runs many iterations in
// one launch:
//   - every CTA of the cluster keeps both clouds (scaled coordinates and
//     column biases in the pair-interleaved layout of k_point.cu) and both
//     state vectors in its own shared memory;
//   - a half-step splits the rows over the CTAs; each row is scored against
//     every column of the other side by S threads (column slices), the
//     partial sums are combined with shuffles;
//   - the new row states are broadcast to every CTA's copy with
//     distributed-shared-memory stores, followed by one cluster barrier.
// Same arithmetic as the streaming kernel ("FlashSinkhorn", Methodologie
// 1-2, in base 2 and the direct form, state L = -kappa f):
//     L_i = log2 sum_j 2^(c_j - kappa |x_i - y_j|^2),  c_j = log2 w_j - Lam_j,
// with the stabiliser m_i = L_old_i + lo, lo the smallest change of any
// column state in the previous half-step (a lower bound of L_new_i - L_old_i,
// so the row sum is >= 1), and an exact two-pass LSE for the first
// half-steps of a launch and for any warp whose sum leaves [2^-80, 2^100).
//
// Control flow is uniform across the cluster (every CTA runs the same number
// of half-steps and barriers, no early exit), so the barriers cannot wait on
// a CTA that left.
#include "common.cuh"
#include "kernels.h"

namespace sot {

constexpr int CL_R = 4;       // rows per thread
constexpr int CL_MAXT = 512;  // threads per CTA at most

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Cluster-wide barrier with release / acquire semantics for shared memory.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store to the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ void cl_store(const float* local_ptr, uint32_t rank, float v) {
    const uint32_t la = (uint32_t)__cvta_generic_to_shared(local_ptr);
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

struct ClusterArgs {
    int B, n, m;
    const float4* xpack;  // [B][n] (x - t, log2 a)
    const float4* ypack;  // [B][m] (y - t, log2 b)
    float* L;             // [B][n] row states, in and out
    float* Lam;           // [B][m]
    float two_kappa;
    int iters;            // full iterations (f-half, then g-half)
    int S;                // threads per row group (column slices), a power of two <= 32
};

// Shared-memory layout of one CTA (floats): image X [ne], image Y [me],
// log2 weights X [n], Y [m], states X [n], Y [m], lo slots [2][8], scratch [32];
// ne = 4 * even(n): pair p of a side holds, as two float4,
//   (-u_2p.x, -u_2p+1.x, -u_2p.y, -u_2p+1.y), (-u_2p.z, -u_2p+1.z, -c_2p, -c_2p+1),
// u = sqrt(kappa) * coordinates, c the column bias of the current half-step.
__host__ __device__ inline int cl_even(int k) { return (k + 1) & ~1; }
size_t cluster_smem_bytes(int n, int m) {
    return sizeof(float) * ((size_t)4 * cl_even(n) + 4 * (size_t)cl_even(m) + 2 * (size_t)n + 2 * (size_t)m + 16 + 32);
}

// One row group's scores against the column pairs p0, p0 + S, ... (< P) of
// image `ic` (the S threads of a group read S adjacent pairs: no bank
// conflicts), rows given by their scaled coordinates (q0, q1, q2 duplicated
// in both lanes).  MODE 0: s_k += 2^(c_j - D - m_k); MODE 1: s_k = max(s_k, c_j - D).
template <int MODE>
__device__ __forceinline__ void cl_rows(const float4* ic, int p0, int S, int P, const float2 (&q0)[CL_R],
                                        const float2 (&q1)[CL_R], const float2 (&q2)[CL_R], const float (&mk)[CL_R],
                                        float (&s)[CL_R]) {
    float2 acc[CL_R];
#pragma unroll
    for (int k = 0; k < CL_R; ++k) acc[k] = MODE ? make_float2(-INFINITY, -INFINITY) : make_float2(0.f, 0.f);
#pragma unroll 2
    for (int pp = p0; pp < P; pp += S) {
        const float4 A = ic[2 * pp], Bv = ic[2 * pp + 1];
        const float2 ncj = make_float2(Bv.z, Bv.w);  // -c
#pragma unroll
        for (int k = 0; k < CL_R; ++k) {
            // base - c + |u - v|^2 with d = u + (-v)
            float2 t = MODE ? ncj : fadd2(make_float2(mk[k], mk[k]), ncj);
            float2 d = fadd2(q0[k], make_float2(A.x, A.y));
            t = ffma2(d, d, t);
            d = fadd2(q1[k], make_float2(A.z, A.w));
            t = ffma2(d, d, t);
            d = fadd2(q2[k], make_float2(Bv.x, Bv.y));
            t = ffma2(d, d, t);
            if (MODE) {
                acc[k].x = fmaxf(acc[k].x, -t.x);
                acc[k].y = fmaxf(acc[k].y, -t.y);
            } else {
                acc[k] = fadd2(acc[k], make_float2(ex2f(-t.x), ex2f(-t.y)));
            }
        }
    }
#pragma unroll
    for (int k = 0; k < CL_R; ++k) s[k] = MODE ? fmaxf(acc[k].x, acc[k].y) : acc[k].x + acc[k].y;
}

__global__ void __launch_bounds__(CL_MAXT) point_cluster_kernel(ClusterArgs a) {
    extern __shared__ float4 cl_smem4[];
    const int b = blockIdx.y;
    const uint32_t rank = cl_rank();
    const int C = (int)gridDim.x;  // one cluster per cloud spans the grid's x dimension
    const int n = a.n, m = a.m;
    const int ne = cl_even(n), me = cl_even(m);
    float4* imgx = cl_smem4;
    float4* imgy = imgx + ne;
    float* w2x = reinterpret_cast<float*>(imgy + me);
    float* w2y = w2x + n;
    float* stx = w2y + m;
    float* sty = stx + n;
    float* loslot = sty + m;  // [2][8]
    float* red = loslot + 16;  // [32]
    const int tid = threadIdx.x, T = blockDim.x;
    const float sk = sqrtf(0.5f * a.two_kappa);

    // ---- load both clouds and both states ------------------------------------------
    auto load_side = [&](const float4* pk, const float* st_in, int N, float4* img, float* w2, float* st) {
        float* f = reinterpret_cast<float*>(img);
        for (int i = tid; i < cl_even(N); i += T) {
            const int pr = i >> 1, k = i & 1;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < N) {
                v = pk[i];
                w2[i] = v.w;
                st[i] = st_in[i];
            }
            f[8 * pr + k] = -__fmul_rn(sk, v.x);
            f[8 * pr + 2 + k] = -__fmul_rn(sk, v.y);
            f[8 * pr + 4 + k] = -__fmul_rn(sk, v.z);
            f[8 * pr + 6 + k] = INFINITY;  // -c; a padding column keeps +inf (score -inf)
        }
    };
    load_side(a.xpack + (size_t)b * n, a.L + (size_t)b * n, n, imgx, w2x, stx);
    load_side(a.ypack + (size_t)b * m, a.Lam + (size_t)b * m, m, imgy, w2y, sty);
    __syncthreads();
    cl_sync();  // every CTA of the cluster exists and is initialised before any remote store

    const int S = a.S;
    const int g = tid / S, sl = tid % S;
    float lo = NAN;  // no bound yet: the first half-step of each side is exact two-pass
    for (int hs = 0; hs < 2 * a.iters; ++hs) {
        const int h = hs & 1;  // 0: f-half (rows X), 1: g-half (rows Y)
        const int nr = h ? m : n, nc = h ? n : m;
        const float4* ir = h ? imgy : imgx;
        float4* ic = h ? imgx : imgy;
        const float* w2c = h ? w2x : w2y;
        const float* stc = h ? stx : sty;
        float* str = h ? sty : stx;
        // column biases of this half-step
        {
            float* f = reinterpret_cast<float*>(ic);
            for (int j = tid; j < nc; j += T) f[8 * (j >> 1) + 6 + (j & 1)] = -__fsub_rn(w2c[j], stc[j]);
        }
        __syncthreads();
        // rows of this CTA, R per thread group
        const int rpc = (nr + C - 1) / C;
        const int rbeg = (int)rank * rpc, rend = min(nr, rbeg + rpc);
        float2 q0[CL_R], q1[CL_R], q2[CL_R];
        float old[CL_R], mk[CL_R], sum[CL_R];
        bool valid[CL_R];
#pragma unroll
        for (int k = 0; k < CL_R; ++k) {
            const int ri = rbeg + g * CL_R + k;
            valid[k] = ri < rend;
            const int rr = valid[k] ? ri : (rbeg < nr ? rbeg : nr - 1);
            const float* f = reinterpret_cast<const float*>(ir) + 8 * (rr >> 1) + (rr & 1);
            const float u0 = -f[0], u1 = -f[2], u2 = -f[4];
            q0[k] = make_float2(u0, u0);
            q1[k] = make_float2(u1, u1);
            q2[k] = make_float2(u2, u2);
            old[k] = valid[k] ? str[ri] : 0.f;
            mk[k] = old[k] + lo;
        }
        const int P = cl_even(nc) >> 1;
        bool exact = !isfinite(lo);
        if (!exact) {
            cl_rows<0>(ic, sl, S, P, q0, q1, q2, mk, sum);
            bool bad = false;
#pragma unroll
            for (int k = 0; k < CL_R; ++k) {
                for (int o = S >> 1; o > 0; o >>= 1) sum[k] += __shfl_xor_sync(0xffffffffu, sum[k], o);
                bad = bad || (valid[k] && !(sum[k] >= SOT_SUM_MIN && sum[k] < SOT_TILE_SUM_MAX));
            }
            exact = __any_sync(0xffffffffu, bad);  // warp-uniform
        }
        if (exact) {
            // two passes: the row maximum, then the sum against it
            float mx[CL_R];
            cl_rows<1>(ic, sl, S, P, q0, q1, q2, mk, mx);
#pragma unroll
            for (int k = 0; k < CL_R; ++k) {
                for (int o = S >> 1; o > 0; o >>= 1) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], o));
                mk[k] = (mx[k] == -INFINITY) ? 0.f : mx[k];
            }
            cl_rows<0>(ic, sl, S, P, q0, q1, q2, mk, sum);
#pragma unroll
            for (int k = 0; k < CL_R; ++k)
                for (int o = S >> 1; o > 0; o >>= 1) sum[k] += __shfl_xor_sync(0xffffffffu, sum[k], o);
        }
        // new states to every copy; the smallest change for the next half-step's bound
        float dmin = INFINITY;
#pragma unroll
        for (int k = 0; k < CL_R; ++k) {
            if (!valid[k]) continue;
            const float nv = mk[k] + log2f(sum[k]);
            dmin = fminf(dmin, old[k] - nv);
            if (sl == 0) {
                const int ri = rbeg + g * CL_R + k;
                for (int q = 0; q < C; ++q) cl_store(str + ri, (uint32_t)q, nv);
            }
        }
        dmin = warp_min(dmin);
        if ((tid & 31) == 0) red[tid >> 5] = dmin;
        __syncthreads();
        if (tid == 0) {
            float v = INFINITY;
            for (int w = 0; w < (T + 31) / 32; ++w) v = fminf(v, red[w]);
            for (int q = 0; q < C; ++q) cl_store(loslot + 8 * (hs & 1) + rank, (uint32_t)q, v);
        }
        cl_sync();
        // every CTA's states and bound contributions are in place
        float v = INFINITY;
        for (int q = 0; q < C; ++q) v = fminf(v, loslot[8 * (hs & 1) + q]);
        lo = (v < INFINITY) ? v : NAN;  // (NaN: no bound, the next half-step is exact)
    }
    // each CTA writes back its own rows of both sides
    {
        const int rpx = (n + C - 1) / C, rpy = (m + C - 1) / C;
        for (int i = (int)rank * rpx + tid; i < min(n, ((int)rank + 1) * rpx); i += T) a.L[(size_t)b * n + i] = stx[i];
        for (int j = (int)rank * rpy + tid; j < min(m, ((int)rank + 1) * rpy); j += T) a.Lam[(size_t)b * m + j] = sty[j];
    }
}

// Plan of a cluster launch for one solve, or false when the problem does not
// qualify (too large for shared memory, or no cluster fits on the device).
bool point_cluster_plan(int B, int n, int m, int sms, int* C_out, int* T_out, int* S_out, size_t* smem_out) {
    if (B < 1 || n < 2 || m < 2) return false;
    const size_t smem = cluster_smem_bytes(n, m);
    if (smem > 200 * 1024) return false;
    int C = 8;
    while (C > 1 && (long long)B * C > 2LL * sms) C >>= 1;
    const int rmax = n > m ? n : m;
    const int rpc = (rmax + C - 1) / C;
    const int groups = (rpc + CL_R - 1) / CL_R;
    if (groups > CL_MAXT) return false;
    int S = 1;
    while (S < 32 && groups * (2 * S) <= CL_MAXT) S <<= 1;
    int T = groups * S;
    T = (T + 31) & ~31;
    if (T > CL_MAXT) return false;
    // Take the cluster path only where it should beat the streaming half-steps:
    // cost models in microseconds per half-step, ~17.4 k pair-evaluations per
    // SM and microsecond either way (the streaming kernel's rate on 2048-point
    // clouds); a streaming half-step adds ~10 us of launch and merge, a cluster
    // half-step ~2 us of barrier and broadcast but uses only B * C / (CTAs per SM)
    // SMs.
    const int cps = (2 * smem <= 227 * 1024 && 2 * T <= 2048) ? 2 : 1;
    double used = (double)B * C / cps;
    if (used > sms) used = sms;
    const double pairs = (double)B * n * m, rate = 17.4e3;
    const double t_cluster = 2.0 + pairs / (used * rate);
    const double t_stream = 10.0 + pairs / ((double)sms * rate);
    if (!(t_cluster < 0.9 * t_stream)) return false;
    *C_out = C;
    *T_out = T;
    *S_out = S;
    *smem_out = smem;
    return true;
}

cudaError_t launch_point_cluster(int B, int n, int m, const float* xpack, const float* ypack, float* L, float* Lam,
                                 float two_kappa, int iters, int C, int T, int S, size_t smem, cudaStream_t st) {
    if (iters <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(point_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ClusterArgs a;
    a.B = B;
    a.n = n;
    a.m = m;
    a.xpack = reinterpret_cast<const float4*>(xpack);
    a.ypack = reinterpret_cast<const float4*>(ypack);
    a.L = L;
    a.Lam = Lam;
    a.two_kappa = two_kappa;
    a.iters = iters;
    a.S = S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, B, 1);
    cfg.blockDim = dim3(T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, point_cluster_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    count_launches(1);
    e = cudaLaunchKernelEx(&cfg, point_cluster_kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sot
