// k_apml.cu -- sparse APML on a stored COO support ("From Theory to
// Throughput: CUDA-Optimized APML", Abstract and Innovation).  With
// s_ij = -C_ij / T on the stored pairs:
//   row softmax R and column softmax K of s over the support,
//   P = (R + K) / 2 (bidirectional symmetrisation),
//   `iters` times: rows scaled to a, then columns scaled to b,
//   loss = sum P_ij C_ij.
//
// The normalisations keep P in factored form, P_ij = U_i S_ij V_j with S the
// symmetrised matrix: scaling the rows of diag(U) S diag(V) to a sets
// U_i = a_i / sum_j S_ij V_j, and scaling its columns to b then sets
// V_j = b_j / sum_i U_i S_ij (a zero sum leaves the factor as it was, as the
// in-place scaling leaves such a row or column alone).  So one normalisation
// reads S and the column indices once (a warp per row: the row sum against
// V, then U_i S_ij added to the column sums from the same, cached, entries),
// and P is written once at the end.
//
// Column quantities (maxima, sums) are gathered per CTA in shared memory and
// written as per-CTA partials that a per-column pass combines in a fixed
// order; with more columns than shared memory holds, the passes add into
// global arrays with atomics instead.  Shared-memory additions run in no fixed
// order: a column's fp32 partial of a few dozen positive terms varies in its
// last bits between runs.  An invalid support is flagged by the first pass and
// reported by the caller; every pass skips column indices out of range, so no
// pass touches memory outside its arrays in the meantime.
#include <algorithm>
#include <climits>

#include "apml.h"
#include "common.cuh"
#include "kernels.h"

namespace sot {

constexpr int AM_T = 256;            // threads of the per-column passes
constexpr int AM_RT = 512;           // threads of the row and entry passes
constexpr int AM_W = AM_RT / 32;     // warps of a row pass
constexpr int AM_R = 8;              // entries of a row a lane holds in registers (one array)
constexpr int AM_R2 = 4;             // the same with two arrays (the last pass)
constexpr int AM_PU = 4;             // entries a thread of the entry pass takes at a time
constexpr int AM_SMEM_COLS = 16384;  // most columns staged (3 floats each in the symmetrisation)

size_t apml_plan(int B, int n, int m, int sms, int* cpc, int* rpc) {
    int c = (2 * std::max(sms, 1) + B - 1) / B;  // about two CTAs per SM in all
    c = std::max(1, std::min(c, (n + 31) / 32));  // at least 32 rows a CTA
    *rpc = (n + c - 1) / c;
    *cpc = (n + *rpc - 1) / *rpc;                // no CTA without rows
    return m <= AM_SMEM_COLS ? (size_t)B * (size_t)*cpc * (size_t)m : 0;
}

// Rows [r0, r1) of this CTA.
__device__ __forceinline__ int apml_rows(const ApmlArgs& p, int* r1) {
    const int r0 = blockIdx.x * p.rpc;
    *r1 = min(p.n, r0 + p.rpc);
    return r0;
}

// Adds v to column j's sum: the CTA's shared partial, or the global fp64 sum.
template <bool SM>
__device__ __forceinline__ void col_add(float* acc, double* csum, int j, float v) {
    if (SM) atomicAdd(acc + j, v);
    else atomicAdd(csum + j, (double)v);
}

// Writes the CTA's shared column partials to part[b][blockIdx.x][:].
__device__ __forceinline__ void flush_partials(const ApmlArgs& p, const float* acc) {
    __syncthreads();
    float* out = p.part + ((size_t)blockIdx.y * p.cpc + blockIdx.x) * p.m;
    for (int j = threadIdx.x; j < p.m; j += AM_RT) out[j] = acc[j];
}

// Per entry: validation, C_ij (direct form), row range markers, column maxima
// of s.  A thread takes AM_PU entries at a time, so that their index loads and
// point gathers are in flight together.
template <bool SM>
__global__ void __launch_bounds__(AM_RT) apml_prep_kernel(ApmlArgs p) {
    extern __shared__ unsigned smax[];
    const int b = blockIdx.y;
    const long long lo_ = p.off[b], hi_ = p.off[b + 1];
    if (lo_ < 0 || hi_ < lo_ || hi_ > p.nnz || (b == 0 && lo_ != 0) || (b == p.B - 1 && hi_ != p.nnz)) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, SOT_DEV_BAD_COO);
        return;  // the cloud's rows keep no range: no later pass reads its entries
    }
    const int lo = (int)lo_, hi = (int)hi_;
    if (SM) {
        for (int j = threadIdx.x; j < p.m; j += AM_RT) smax[j] = 0u;
        __syncthreads();
    }
    const float* Xb = p.X + (size_t)b * p.n * p.d;
    const float* Yb = p.Y + (size_t)b * p.m * p.d;
    unsigned* gmax = p.cmax + (size_t)b * p.m;
    const int chunk = (int)((hi - lo + (long long)gridDim.x - 1) / gridDim.x);
    const int c0 = lo + (int)blockIdx.x * chunk, c1 = (int)min((long long)hi, (long long)c0 + chunk);
    for (int eb = c0 + threadIdx.x; eb < c1; eb += AM_RT * AM_PU) {
        int iv[AM_PU], jv[AM_PU], ip[AM_PU], in[AM_PU];
#pragma unroll
        for (int u = 0; u < AM_PU; ++u) {
            const int e = eb + AM_RT * u;
            iv[u] = -1;
            jv[u] = -1;
            ip[u] = -1;
            in[u] = INT_MAX;
            if (e < c1) {
                iv[u] = __ldg(p.rows + e);
                jv[u] = __ldg(p.cols + e);
                if (e > lo) ip[u] = __ldg(p.rows + e - 1);
                if (e + 1 < hi) in[u] = __ldg(p.rows + e + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < AM_PU; ++u) {
            const int e = eb + AM_RT * u;
            if (e >= c1) continue;
            const int i = iv[u], j = jv[u];
            if (i < 0 || i >= p.n || j < 0 || j >= p.m || in[u] < i) {
                atomicOr(p.status, SOT_DEV_BAD_COO);
                continue;
            }
            const float* x = Xb + (size_t)i * p.d;
            const float* y = Yb + (size_t)j * p.d;
            float c = 0.f;
            for (int k = 0; k < p.d; ++k) {
                const float t = __ldg(x + k) - __ldg(y + k);
                c = fmaf(t, t, c);
            }
            p.cost[e] = c;
            // entries of row i are [rstart, rend) relative to the cloud's first entry + 1
            if (ip[u] != i) p.rstart[(size_t)b * p.n + i] = (int)(e - lo) + 1;
            if (in[u] != i) p.rend[(size_t)b * p.n + i] = (int)(e - lo) + 1;
            const unsigned key = ord_encode(-c * p.inv_T);
            if (SM) atomicMax(smax + j, key);
            else atomicMax(gmax + j, key);
        }
    }
    if (SM) {
        __syncthreads();
        unsigned* out = reinterpret_cast<unsigned*>(p.part) + ((size_t)b * p.cpc + blockIdx.x) * p.m;
        for (int j = threadIdx.x; j < p.m; j += AM_RT) out[j] = smax[j];
    }
}

// Per column: the maximum of s (a column without entries is never read).
template <bool SM>
__global__ void apml_colmax_kernel(ApmlArgs p) {
    const long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (c >= (long long)p.B * p.m) return;
    unsigned v = 0u;
    if (SM) {
        const long long b = c / p.m, j = c - b * p.m;
        const unsigned* in = reinterpret_cast<const unsigned*>(p.part) + (size_t)b * p.cpc * p.m + j;
#pragma unroll 8
        for (int k = 0; k < p.cpc; ++k) v = max(v, in[(size_t)k * p.m]);
    } else {
        v = p.cmax[c];
    }
    p.cm[c] = v ? ord_decode(v) : 0.f;
}

// Per column: combines the partial sums.  mode 0: cfac = 1 / sum (softmax
// exponentials); mode 1: V_j = b_j / sum (`first`: the previous V is 1).  The
// partials are added in fp32 with an error-free transformation of each
// addition (two-sum, Knuth) and the rounding errors carried along, which keeps
// the sum within about an ulp of the exact one at the fp32 pipe's rate (this
// GPU's fp64 rate is low enough to dominate the pass).
template <bool SM>
__global__ void apml_colfactor_kernel(ApmlArgs p, int mode, int first) {
    const long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (c >= (long long)p.B * p.m) return;
    float cs;
    if (SM) {
        const long long b = c / p.m, j = c - b * p.m;
        const float* in = p.part + (size_t)b * p.cpc * p.m + j;
        float s = 0.f, err = 0.f;
#pragma unroll 8
        for (int k = 0; k < p.cpc; ++k) {
            const float x = in[(size_t)k * p.m];
            const float t = s + x, z = t - s;
            err += (s - (t - z)) + (x - z);
            s = t;
        }
        cs = s + err;
    } else {
        cs = (float)p.csum[c];
        p.csum[c] = 0.0;  // ready for the next pass
    }
    if (mode == 0) {
        p.cfac[c] = cs > 0.f ? 1.f / cs : 0.f;
    } else {
        const float bj = p.b ? p.b[c] : 1.f / (float)p.m;
        if (cs > 0.f) p.vfac[c] = bj / cs;
        else if (first) p.vfac[c] = 1.f;
    }
}

// Stages [B][m] column values of cloud blockIdx.y into shared memory.
__device__ __forceinline__ void stage_cols(float* dst, const float* src, int m) {
    const float* s = src + (size_t)blockIdx.y * m;
    for (int j = threadIdx.x; j < m; j += AM_RT) dst[j] = s[j];
}

__device__ __forceinline__ void zero_cols(float* dst, int m) {
    for (int j = threadIdx.x; j < m; j += AM_RT) dst[j] = 0.f;
}

// ---- row passes -------------------------------------------------------------
// A warp takes the rows i = r0 + w + AM_W k of its CTA.  Per group of 32 rows,
// lane k loads row k's entry range and a float4 of per-row data up front; a
// row's first 32 R entries are held in registers (R per lane), loaded while
// the previous row is processed; a longer row's further entries are loaded one
// at a time.  A lane holds the entries s0 + lane + 32 u.  Entry indices fit in
// an int (the caller bounds nnz below 2^31).

template <int R, int NA>
struct Chunk {
    float v[NA][R];  // v[0]: first array, v[NA - 1]: second
    int j[R];        // column, -1 for no entry (or an index out of range)
};

__device__ __forceinline__ int col_or_none(const int* cols, int e, int m) {
    const int j = __ldg(cols + e);
    return (unsigned)j < (unsigned)m ? j : -1;
}

template <int R, int NA>
__device__ __forceinline__ void load_chunk(Chunk<R, NA>& c, const float* a0, const float* a1, const int* cols, int m,
                                           int e0, int s1) {
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int e = e0 + 32 * u;
        c.j[u] = -1;
        c.v[0][u] = 0.f;
        c.v[NA - 1][u] = 0.f;
        if (e < s1) {
            c.j[u] = col_or_none(cols, e, m);
            c.v[0][u] = __ldg(a0 + e);
            if (NA > 1) c.v[NA - 1][u] = __ldg(a1 + e);
        }
    }
}

// fn(v0, v1, j, e) on the chunk's entries, then on the rest of the row [s0, s1)
// one entry at a time (NC: a0 is read-only during the kernel; otherwise the
// lane re-reads values it wrote, with coherent loads).  fn may change v0; the
// chunk keeps the new value.
template <bool NC = true, int R, int NA, class F>
__device__ __forceinline__ void each_entry(Chunk<R, NA>& c, int s0, int s1, const float* a0, const float* a1,
                                           const int* cols, int m, F&& fn) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < R; ++u)
        if (c.j[u] >= 0) fn(c.v[0][u], c.v[NA - 1][u], c.j[u], s0 + lane + 32 * u);
    for (int e = s0 + 32 * R + lane; e < s1; e += 32) {
        const int j = col_or_none(cols, e, m);
        if (j < 0) continue;
        float v0 = NC ? __ldg(a0 + e) : a0[e];
        float v1 = NA > 1 ? __ldg(a1 + e) : 0.f;
        fn(v0, v1, j, e);
    }
}

// Runs body(i, s0, s1, x, chunk) for the warp's rows in order (s0 == s1 for a
// row without entries); extra(i) gives the row's float4 of per-row data.
template <int R, int NA, class Extra, class Body>
__device__ __forceinline__ void row_pass(const ApmlArgs& p, const float* a0, const float* a1, Extra&& extra,
                                         Body&& body) {
    const int b = blockIdx.y, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int r1;
    const int first = apml_rows(p, &r1) + w;
    const int nk = first < r1 ? (r1 - first + AM_W - 1) / AM_W : 0;
    const int base = (int)p.off[b];
    for (int kb = 0; kb < nk; kb += 32) {
        const int kn = min(32, nk - kb);
        // lane k: row kb + k's entries [st, en) and per-row data
        int st = base, en = base;
        float4 xt = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane < kn) {
            const int i = first + AM_W * (kb + lane);
            const size_t ri = (size_t)b * p.n + i;
            const int rs = p.rstart[ri];
            if (rs) {
                st = base + rs - 1;
                en = base + p.rend[ri];
            }
            xt = extra(i);
        }
        Chunk<R, NA> cur, nxt;
        load_chunk(cur, a0, a1, p.cols, p.m, __shfl_sync(0xffffffffu, st, 0) + lane, __shfl_sync(0xffffffffu, en, 0));
        for (int k = 0; k < kn; ++k) {
            const int s0 = __shfl_sync(0xffffffffu, st, k), s1 = __shfl_sync(0xffffffffu, en, k);
            const float4 x = make_float4(__shfl_sync(0xffffffffu, xt.x, k), __shfl_sync(0xffffffffu, xt.y, k),
                                         __shfl_sync(0xffffffffu, xt.z, k), __shfl_sync(0xffffffffu, xt.w, k));
            const int kx = min(k + 1, 31);
            const int n0 = __shfl_sync(0xffffffffu, st, kx), n1 = __shfl_sync(0xffffffffu, en, kx);
            if (k + 1 < kn) load_chunk(nxt, a0, a1, p.cols, p.m, n0 + lane, n1);
            body(first + AM_W * (kb + k), s0, s1, x, cur);
            cur = nxt;
        }
    }
}

// Row softmax statistics (maximum of s, sum of exp(s - maximum)); the column
// softmax's exponentials exp(s_ij - max_i' s_i'j) go to the column sums.
template <bool SM>
__global__ void __launch_bounds__(AM_RT, 2) apml_rowstat_kernel(ApmlArgs p) {
    extern __shared__ float sh[];
    const int b = blockIdx.y, lane = threadIdx.x & 31;
    float* scm = sh;
    float* acc = sh + p.m;
    if (SM) {
        stage_cols(scm, p.cm, p.m);
        zero_cols(acc, p.m);
        __syncthreads();
    }
    const float* cmv = SM ? scm : p.cm + (size_t)b * p.m;
    double* cs = p.csum + (size_t)b * p.m;
    const float it = p.inv_T;
    row_pass<AM_R, 1>(p, p.cost, nullptr, [](int) { return make_float4(0.f, 0.f, 0.f, 0.f); },
                [&](int i, int s0, int s1, float4, Chunk<AM_R, 1>& c) {
                    if (s0 == s1) return;
                    float mx = -INFINITY;
                    each_entry(c, s0, s1, p.cost, nullptr, p.cols, p.m, [&](float& cv, float&, int j, int) {
                        const float s = -cv * it;
                        mx = fmaxf(mx, s);
                        col_add<SM>(acc, cs, j, expf(s - cmv[j]));
                    });
                    mx = warp_max(mx);
                    float sm = 0.f;
                    each_entry(c, s0, s1, p.cost, nullptr, p.cols, p.m,
                                  [&](float& cv, float&, int, int) { sm += expf(-cv * it - mx); });
                    sm = warp_sum(sm);
                    if (lane == 0) p.rstat[(size_t)b * p.n + i] = make_float2(mx, sm);
                });
    if (SM) flush_partials(p, acc);
}

// S = (R + K) / 2 into vals; with normalisations to follow, also the first row
// scaling (V = 1): U_i = a_i / sum_j S_ij, and U_i S_ij added to the column sums.
template <bool SM>
__global__ void __launch_bounds__(AM_RT, 2) apml_sym_kernel(ApmlArgs p) {
    extern __shared__ float sh[];
    const int b = blockIdx.y, lane = threadIdx.x & 31;
    float* scm = sh;
    float* scf = sh + p.m;
    float* acc = sh + 2 * p.m;
    const bool norm = p.iters > 0;
    if (SM) {
        stage_cols(scm, p.cm, p.m);
        stage_cols(scf, p.cfac, p.m);
        if (norm) zero_cols(acc, p.m);
        __syncthreads();
    }
    const float* cmv = SM ? scm : p.cm + (size_t)b * p.m;
    const float* cfv = SM ? scf : p.cfac + (size_t)b * p.m;
    double* cs = p.csum + (size_t)b * p.m;
    const float it = p.inv_T, an = 1.f / (float)p.n;
    row_pass<AM_R, 1>(p, p.cost, nullptr,
                [&](int i) {
                    const size_t ri = (size_t)b * p.n + i;
                    const float2 r = p.rstat[ri];
                    return make_float4(r.x, r.y, p.a ? p.a[ri] : an, 0.f);
                },
                [&](int i, int s0, int s1, float4 x, Chunk<AM_R, 1>& c) {
                    if (s0 == s1) return;
                    float tot = 0.f;
                    // the chunk's values become S_ij (kept for the scatter below)
                    each_entry(c, s0, s1, p.cost, nullptr, p.cols, p.m, [&](float& cv, float&, int j, int e) {
                        const float s = -cv * it;
                        const float r = expf(s - x.x) / x.y;
                        const float k = expf(s - cmv[j]) * cfv[j];
                        const float v = 0.5f * (r + k);
                        p.vals[e] = v;
                        tot += v;
                        cv = v;
                    });
                    if (!norm) return;
                    tot = warp_sum(tot);
                    const float uf = tot > 0.f ? x.z / tot : 1.f;
                    if (lane == 0) p.ufac[(size_t)b * p.n + i] = uf;
                    // beyond the first chunk, the lane re-reads the values it wrote (coherent loads)
                    each_entry<false>(c, s0, s1, p.vals, nullptr, p.cols, p.m,
                                         [&](float& v, float&, int j, int) { col_add<SM>(acc, cs, j, uf * v); });
                });
    if (SM && norm) flush_partials(p, acc);
}

// One row scaling against the current V: U_i = a_i / sum_j S_ij V_j, then
// U_i S_ij added to the column sums.
template <bool SM>
__global__ void __launch_bounds__(AM_RT, 2) apml_rownorm_kernel(ApmlArgs p) {
    extern __shared__ float sh[];
    const int b = blockIdx.y, lane = threadIdx.x & 31;
    float* sv = sh;
    float* acc = sh + p.m;
    if (SM) {
        stage_cols(sv, p.vfac, p.m);
        zero_cols(acc, p.m);
        __syncthreads();
    }
    const float* vv = SM ? sv : p.vfac + (size_t)b * p.m;
    double* cs = p.csum + (size_t)b * p.m;
    const float an = 1.f / (float)p.n;
    row_pass<AM_R, 1>(p, p.vals, nullptr,
                [&](int i) {
                    const size_t ri = (size_t)b * p.n + i;
                    return make_float4(p.a ? p.a[ri] : an, p.ufac[ri], 0.f, 0.f);
                },
                [&](int i, int s0, int s1, float4 x, Chunk<AM_R, 1>& c) {
                    if (s0 == s1) return;
                    float tot = 0.f;
                    each_entry(c, s0, s1, p.vals, nullptr, p.cols, p.m,
                                  [&](float& k, float&, int j, int) { tot = fmaf(k, vv[j], tot); });
                    tot = warp_sum(tot);
                    const float uf = tot > 0.f ? x.x / tot : x.y;
                    if (lane == 0) p.ufac[(size_t)b * p.n + i] = uf;
                    each_entry(c, s0, s1, p.vals, nullptr, p.cols, p.m,
                                  [&](float& k, float&, int j, int) { col_add<SM>(acc, cs, j, uf * k); });
                });
    if (SM) flush_partials(p, acc);
}

// P_ij = U_i S_ij V_j written over S (after normalisations), the per-row
// loss terms sum_j P_ij C_ij and, for d <= 3, the support gradient
// 2 sum_j P_ij (x_i - y_j) (both in a fixed order).
template <bool SM>
__global__ void __launch_bounds__(AM_RT, 2) apml_final_kernel(ApmlArgs p) {
    extern __shared__ float sh[];
    const int b = blockIdx.y, lane = threadIdx.x & 31;
    const bool norm = p.iters > 0;
    if (SM && norm) {
        stage_cols(sh, p.vfac, p.m);
        __syncthreads();
    }
    const float* vv = SM ? sh : p.vfac + (size_t)b * p.m;
    const int d = p.d;
    const float* yb = p.Y + (size_t)b * p.m * d;
    row_pass<AM_R2, 2>(p, p.vals, p.cost,
                       [&](int i) {
                           const float* xi = p.X + ((size_t)b * p.n + i) * d;
                           return make_float4(norm ? p.ufac[(size_t)b * p.n + i] : 1.f, xi[0], d > 1 ? xi[1] : 0.f,
                                              d > 2 ? xi[2] : 0.f);
                       },
                       [&](int i, int s0, int s1, float4 x, Chunk<AM_R2, 2>& c) {
                    float l = 0.f, g0 = 0.f, g1 = 0.f, g2 = 0.f;
                    each_entry(c, s0, s1, p.vals, p.cost, p.cols, p.m, [&](float& k, float& cv, int j, int e) {
                        float v = k;
                        if (norm) {
                            v = x.x * k * vv[j];
                            p.vals[e] = v;
                        }
                        l = fmaf(v, cv, l);
                        if (p.grad) {
                            const float* y = yb + (size_t)j * d;
                            g0 = fmaf(v, x.y - __ldg(y), g0);
                            if (d > 1) g1 = fmaf(v, x.z - __ldg(y + 1), g1);
                            if (d > 2) g2 = fmaf(v, x.w - __ldg(y + 2), g2);
                        }
                    });
                    l = warp_sum(l);
                    if (lane == 0) p.loss_part[(size_t)b * p.n + i] = l;
                    if (p.grad) {
                        g0 = warp_sum(g0);
                        g1 = warp_sum(g1);
                        g2 = warp_sum(g2);
                        if (lane == 0) {
                            float* gi = p.grad + ((size_t)b * p.n + i) * d;
                            gi[0] = 2.f * g0;
                            if (d > 1) gi[1] = 2.f * g1;
                            if (d > 2) gi[2] = 2.f * g2;
                        }
                    }
                });
}

template <bool SM>
static cudaError_t run_apml(const ApmlArgs& p, cudaStream_t st) {
    const int m = p.m;
    const dim3 gr(p.cpc, p.B);
    const unsigned gf = (unsigned)(((long long)p.B * m + AM_T - 1) / AM_T);
    const size_t s1 = SM ? sizeof(float) * m : 0, s2 = 2 * s1, s3 = 3 * s1;
    if (SM) {
        cudaError_t e = cudaFuncSetAttribute(apml_sym_kernel<SM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(apml_rowstat_kernel<SM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(apml_rownorm_kernel<SM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(apml_prep_kernel<SM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(apml_final_kernel<SM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
        if (e != cudaSuccess) return e;
    }
    count_launches(6 + 2 * std::max(p.iters - 1, 0) + (p.iters > 0 ? 1 : 0));
    apml_prep_kernel<SM><<<gr, AM_RT, s1, st>>>(p);
    apml_colmax_kernel<SM><<<gf, AM_T, 0, st>>>(p);
    apml_rowstat_kernel<SM><<<gr, AM_RT, s2, st>>>(p);
    apml_colfactor_kernel<SM><<<gf, AM_T, 0, st>>>(p, 0, 0);
    apml_sym_kernel<SM><<<gr, AM_RT, p.iters > 0 ? s3 : s2, st>>>(p);
    for (int it = 0; it < p.iters; ++it) {
        apml_colfactor_kernel<SM><<<gf, AM_T, 0, st>>>(p, 1, it == 0);
        if (it + 1 < p.iters) apml_rownorm_kernel<SM><<<gr, AM_RT, s2, st>>>(p);
    }
    apml_final_kernel<SM><<<gr, AM_RT, p.iters > 0 ? s1 : 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_apml(const ApmlArgs& p, cudaStream_t st) {
    if (p.B < 1 || p.n < 1 || p.m < 1 || p.d < 1 || !(p.inv_T > 0.f) || p.iters < 0 || p.cpc < 1 || p.rpc < 1 ||
        (long long)p.cpc * p.rpc < p.n || (p.grad && p.d > 3))
        return cudaErrorInvalidValue;
    const bool sm = p.part != nullptr;
    if (sm && p.m > AM_SMEM_COLS) return cudaErrorInvalidValue;
    cudaError_t e = sm ? run_apml<true>(p, st) : run_apml<false>(p, st);
    if (e != cudaSuccess || !p.loss) return e;
    return launch_reduce_parts(p.loss_part, p.B, p.n, p.loss, st);
}

}  // namespace sot
