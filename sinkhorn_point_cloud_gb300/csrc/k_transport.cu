// k_transport.cu -- transport-matrix products P V streamed without storing P
// ("FlashSinkhorn", Methodologie 3: the plan is applied as an attention-like
// weighted sum; its HVP paragraph builds the Hessian-vector product from
// such transport-vector and transport-matrix products).
//
// One thread per row.  Column tiles (coordinates transposed, so that a row
// value is reused by a group of W columns: 8 when d > 8, 4 in the low
// dimensions, where the exact evaluation and not the screen dominates) and the
// tile's V rows sit in shared memory.  Columns are split into chunks so that
// the grid fills the SMs; a second kernel adds the chunks' partial sums in
// chunk order (deterministic).
//
// Each pair is first scored in fp32 in the direct form: log2(P_ij / w_i) is
// about log2 w'_j + kappa (f_i + g_j - C_ij).  A pair below -(26 + log2 nc) - 4 is
// skipped: its weight is under 2^-30 / nc of w_i, so all skipped pairs of a row
// together carry less than 2^-30 of it (the 4 units cover the fp32 estimate's
// own error many times over), far below fp32 resolution of the sum.  The test
// is taken as C_ij < f_i + h_j with the column's limit
// h_j = g_j + (log2 w'_j + 30 + log2 nc) / kappa staged with the tile.  Every
// other pair is evaluated exactly: C_ij from error-free coordinate differences
// and squares in float-float, and the exponent, where the potentials and C_ij
// cancel to a small number, in float-float throughout (the fp64 pipe is slow
// on this part).
//
// The exact evaluations are shared out over the warp: per block of columns
// (the whole tile when d <= 8, where they dominate; 8 columns above, where the
// screen does and shared memory is scarcer), the pairs its 32 rows' screens
// passed are queued in shared memory (row by row, each row's in column order)
// and evaluated one per lane, so a column that matters to one row of a warp
// costs one lane, not the warp.  Each row then adds its pairs' terms in
// column order, as a serial loop over the columns would.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "transport.h"

namespace sot {

constexpr int TR_T = 128;        // rows per CTA (one per thread)
constexpr int TR_CT = 32;        // columns per shared-memory tile
constexpr int TR_YS = TR_CT + 4; // its row stride (keeps float4 reads aligned; 4-way store conflicts, not 32)
constexpr int TR_VS = TR_CT + 1; // row stride of the tile's V values, transposed (rows read at 32 columns at once)
constexpr int TR_MAXD = 256;
constexpr int TR_MAXC = 64;

int transport_max_d() { return TR_MAXD; }
int transport_max_c() { return TR_MAXC; }

// row stride of the row tile in shared memory: odd, so the 32 rows of a warp
// fall in 32 different banks
__host__ __device__ inline int tr_ldx(int d) { return (d % 2 == 0) ? d + 1 : d; }

// column group of the screen (one row value reused by W columns) and columns
// per exact-evaluation queue
__host__ __device__ constexpr int tr_w(int d) { return d > 8 ? 8 : 4; }
__host__ __device__ constexpr int tr_qg(int w) { return w == 8 ? 8 : TR_CT; }

static size_t tr_smem_bytes(int d, int c) {
    return sizeof(float) * ((size_t)TR_T * tr_ldx(d) + (size_t)d * TR_YS + 3 * TR_CT + 2 * TR_T + (size_t)TR_VS * c +
                            (size_t)TR_T * tr_qg(tr_w(d)));
}

// CENTRED (row-centred products for the Hessian-vector product, d <= TR_CD):
// per row i, with yhat_i = p.rc[i] and v_i = p.rv[i] (both [d]) and the
// column values g_j = V[j][0] (c = 1), out[i] = [ sum_j w_ij ((y_j - yhat_i).v_i)(y_j - yhat_i),
// sum_j w_ij g_j (y_j - yhat_i) ] (2d values): the differences are formed per
// pair, so no two large sums cancel.
constexpr int TR_CD = 9;

// DF: the number of coordinates fixed at compile time (0: p.d at run time).
template <int CV, int W, bool CENTRED = false, int DF = 0>
__global__ void __launch_bounds__(TR_T) transport_kernel(TransportArgs p) {
    static_assert(W == 4 || W == 8, "column group of 4 or 8");
    static_assert(DF >= 0 && DF <= 8, "fixed dimension of at most 8");
    extern __shared__ float smem[];
    const int d = DF ? DF : p.d, c = p.c, ldx = tr_ldx(d);
    float* xs = smem;                 // [TR_T][ldx] this CTA's rows
    float* ys = xs + TR_T * ldx;      // [d][TR_YS] column tile, transposed and negated
    float* hs = ys + d * TR_YS;       // [TR_CT] screen limits h_j (-inf past the end; float4 reads)
    float2* bs = reinterpret_cast<float2*>(hs + TR_CT);  // [TR_CT] kappa g_j + log2 w'_j (float-float)
    float2* as = bs + TR_CT;          // [TR_T] kappa f_i + log2 w_i (float-float)
    float* vs = reinterpret_cast<float*>(as + TR_T);  // [c][TR_VS] V values of the tile, transposed
    constexpr int QG = tr_qg(W);
    unsigned* qs = reinterpret_cast<unsigned*>(vs + TR_VS * c);  // [TR_T / 32][32 QG] per-warp pair queues
    const int lane = threadIdx.x & 31, wrp = threadIdx.x >> 5;
    unsigned* q = qs + wrp * (32 * QG);  // entries (row lane << 5 | column), then their weights
    float* qw = reinterpret_cast<float*>(q);
    const int b = blockIdx.y;
    const int rb = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rb * TR_T;
    const int c_begin = ch * p.chunk, c_end = min(p.nc, c_begin + p.chunk);
    const int i = row0 + threadIdx.x;
    const bool ok = i < p.nr;
    const float* R = p.R + (size_t)b * p.nr * d;
    const float* Cl = p.Cl + (size_t)b * p.nc * d;
    const float* Vb = p.V + (size_t)b * p.nc * p.ldv;

    for (int e = threadIdx.x; e < TR_T * d; e += TR_T) {
        const int r = e / d, k = e % d;
        xs[r * ldx + k] = (row0 + r < p.nr) ? R[(size_t)(row0 + r) * d + k] : 0.f;
    }
    const float2 kap = make_float2(p.kap_hi, p.kap_lo);
    const float fi = ok ? p.fr[(size_t)b * p.nr + i] : 0.f;
    {
        const float lwi = ok ? (p.wr ? log2f(p.wr[(size_t)b * p.nr + i]) : -log2f((float)p.nr)) : 0.f;
        as[threadIdx.x] = ff_add(ff_mul(kap, make_float2(fi, 0.f)), make_float2(lwi, 0.f));
    }
    const float sig = -(30.f + log2f((float)p.nc));  // skip threshold on log2(P_ij / w_i)
    // a fixed small dimension keeps the row in registers, each value paired for the packed screen
    float2 xp[DF ? DF : 1];
    if (DF) {
#pragma unroll
        for (int k = 0; k < (DF ? DF : 1); ++k) {
            const float x = ok ? R[(size_t)i * d + k] : 0.f;
            xp[k] = make_float2(x, x);
        }
    }
    float acc[CV];
#pragma unroll
    for (int k = 0; k < CV; ++k) acc[k] = 0.f;
    const float* xr = xs + threadIdx.x * ldx;
    // centred mode: the row's barycentre and direction, and the two sums
    float yh[CENTRED ? TR_CD : 1], vr[CENTRED ? TR_CD : 1], aco[CENTRED ? TR_CD : 1], agy[CENTRED ? TR_CD : 1];
    if (CENTRED) {
#pragma unroll
        for (int k = 0; k < TR_CD; ++k) {
            const bool kk = ok && k < d;
            yh[k] = kk ? p.rc[((size_t)b * p.nr + i) * d + k] : 0.f;
            vr[k] = kk ? p.rv[((size_t)b * p.nr + i) * d + k] : 0.f;
            aco[k] = 0.f;
            agy[k] = 0.f;
        }
    }

    for (int base = c_begin; base < c_end; base += TR_CT) {
        __syncthreads();
        // coalesced reads of whole column rows (the transposed stores are 4-way
        // bank conflicts with the padded stride)
        for (int e = threadIdx.x; e < TR_CT * d; e += TR_T) {
            const int jj = e / d, k = e % d, j = base + jj;
            ys[k * TR_YS + jj] = (j < c_end) ? -Cl[(size_t)j * d + k] : 0.f;  // negated
        }
        for (int e = threadIdx.x; e < TR_CT * c; e += TR_T) {
            const int jj = e / c, k = e % c, j = base + jj;
            vs[k * TR_VS + jj] = (j < c_end) ? Vb[(size_t)j * p.ldv + k] : 0.f;
        }
        if (threadIdx.x < TR_CT) {
            const int j = base + threadIdx.x;
            const bool cj = j < c_end;
            const float gj = cj ? p.gc[(size_t)b * p.nc + j] : 0.f;
            const float lj = cj ? (p.wc ? log2f(p.wc[(size_t)b * p.nc + j]) : -log2f((float)p.nc)) : 0.f;
            hs[threadIdx.x] = cj ? gj + (lj - sig) / p.kap_hi : -INFINITY;
            bs[threadIdx.x] = ff_add(ff_mul(kap, make_float2(gj, 0.f)), make_float2(lj, 0.f));
        }
        __syncthreads();
        for (int qb = 0; qb < TR_CT; qb += QG) {
            // screen: bit jj of `sm` is set when pair (i, base + jj) needs its exact weight
            unsigned sm = 0;
            if (ok) {
                for (int jg = qb; jg < qb + QG; jg += W) {
                    // fp32 direct-form distances of W columns less f_i, two per packed instruction
                    float2 cp[W / 2];
#pragma unroll
                    for (int h = 0; h < W / 2; ++h) cp[h] = make_float2(-fi, -fi);
                    if (DF) {
#pragma unroll
                        for (int k = 0; k < (DF ? DF : 1); ++k) {
#pragma unroll
                            for (int qq = 0; qq < W / 4; ++qq) {
                                const float4 y4 = *reinterpret_cast<const float4*>(ys + k * TR_YS + jg + 4 * qq);
                                const float2 t0 = fadd2(xp[k], make_float2(y4.x, y4.y));
                                const float2 t1 = fadd2(xp[k], make_float2(y4.z, y4.w));
                                cp[2 * qq] = ffma2(t0, t0, cp[2 * qq]);
                                cp[2 * qq + 1] = ffma2(t1, t1, cp[2 * qq + 1]);
                            }
                        }
                    } else {
                        // the next coordinate's values are loaded while this one's are
                        // used (the loads one past the last coordinate stay inside the
                        // shared arrays and are not used)
                        float xn = xr[0];
                        float4 yn[W / 4];
#pragma unroll
                        for (int qq = 0; qq < W / 4; ++qq)
                            yn[qq] = *reinterpret_cast<const float4*>(ys + jg + 4 * qq);
#pragma unroll 4
                        for (int k = 0; k < d; ++k) {
                            const float2 xx = make_float2(xn, xn);
                            float4 yc[W / 4];
#pragma unroll
                            for (int qq = 0; qq < W / 4; ++qq) {
                                yc[qq] = yn[qq];
                                yn[qq] = *reinterpret_cast<const float4*>(ys + (k + 1) * TR_YS + jg + 4 * qq);
                            }
                            xn = xr[k + 1];
#pragma unroll
                            for (int qq = 0; qq < W / 4; ++qq) {
                                const float2 t0 = fadd2(xx, make_float2(yc[qq].x, yc[qq].y));
                                const float2 t1 = fadd2(xx, make_float2(yc[qq].z, yc[qq].w));
                                cp[2 * qq] = ffma2(t0, t0, cp[2 * qq]);
                                cp[2 * qq + 1] = ffma2(t1, t1, cp[2 * qq + 1]);
                            }
                        }
                    }
#pragma unroll
                    for (int qq = 0; qq < W / 4; ++qq) {
                        // the screen in fp32: C_ij - f_i < h_j
                        const float4 h4 = *reinterpret_cast<const float4*>(hs + jg + 4 * qq);
                        const int u = jg + 4 * qq - qb;
                        sm |= (cp[2 * qq].x < h4.x ? 1u : 0u) << u;
                        sm |= (cp[2 * qq].y < h4.y ? 2u : 0u) << u;
                        sm |= (cp[2 * qq + 1].x < h4.z ? 4u : 0u) << u;
                        sm |= (cp[2 * qq + 1].y < h4.w ? 8u : 0u) << u;
                    }
                }
            }
            // queue the warp's pairs of this block: this lane's run starts at `o`
            const int cnt = __popc(sm);
            int o = cnt;
#pragma unroll
            for (int s = 1; s < 32; s <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, o, s);
                if (lane >= s) o += t;
            }
            const int total = __shfl_sync(0xffffffffu, o, 31);
            o -= cnt;
            if (total == 0) continue;  // warp-uniform
            {
                int k = o;
                for (unsigned mm = sm; mm; mm &= mm - 1)
                    q[k++] = ((unsigned)lane << 5) | (unsigned)(qb + __ffs(mm) - 1);
            }
            __syncwarp();
            // exact weights, one queued pair per lane: C_ij from exact differences
            // and squares (positive terms: their high parts added error-free, the
            // low parts in fp32), then
            // log2 P_ij = (kappa f_i + log2 w_i) + (kappa g_j + log2 w'_j) - kappa C_ij,
            // all in float-float
            for (int t = lane; t < total; t += 32) {
                const unsigned e = q[t];
                const int jj = (int)(e & 31u), r = (wrp << 5) | (int)(e >> 5);
                const float* xq = xs + r * ldx;
                // NC independent sums (coordinates k = u mod NC) when d is only known
                // at run time, so that a long row is not one chain of dependent adds
                // (one with 64 accumulators per row, which leave no registers for more)
                constexpr int NC = (DF || CV > 16) ? 1 : 4;
                float chi[NC], clo[NC];
#pragma unroll
                for (int u = 0; u < NC; ++u) chi[u] = clo[u] = 0.f;
                for (int k0 = 0; k0 < d; k0 += NC) {
#pragma unroll
                    for (int u = 0; u < NC; ++u) {
                        const int k = k0 + u;
                        if (NC == 1 || k < d) {
                            const float2 dd = two_sum(xq[k], ys[k * TR_YS + jj]);
                            const float2 sq = two_prod(dd.x, dd.x);
                            const float2 sh = two_sum(chi[u], sq.x);
                            chi[u] = sh.x;
                            clo[u] = __fadd_rn(clo[u], __fadd_rn(sh.y, __fmaf_rn(__fadd_rn(dd.x, dd.x), dd.y, sq.y)));
                        }
                    }
                }
                float2 C2 = ff_renorm(chi[0], clo[0]);
#pragma unroll
                for (int u = 1; u < NC; ++u) C2 = ff_add(C2, ff_renorm(chi[u], clo[u]));
                const float2 kc = ff_mul(kap, C2);
                const float2 ell = ff_add(ff_add(as[r], bs[jj]), make_float2(-kc.x, -kc.y));
                qw[t] = exp2f(__fadd_rn(ell.x, ell.y));
            }
            __syncwarp();
            // this row's terms, in column order
            {
                int k = o;
                for (unsigned mm = sm; mm; mm &= mm - 1, ++k) {
                    const int jj = qb + __ffs(mm) - 1;
                    const float w = qw[k];
                    const float* vj = vs + jj;  // V_j[k] at vj[k TR_VS]
                    if (CENTRED) {
                        // y_j - yhat_i (the tile holds -y_j), its projection on v_i
                        float dk[TR_CD], dv = 0.f;
#pragma unroll
                        for (int kk = 0; kk < TR_CD; ++kk) {
                            dk[kk] = (kk < d) ? -ys[kk * TR_YS + jj] - yh[kk] : 0.f;
                            dv = fmaf(dk[kk], vr[kk], dv);
                        }
                        const float wdv = w * dv, wg = w * vj[0];
#pragma unroll
                        for (int kk = 0; kk < TR_CD; ++kk) {
                            aco[kk] = fmaf(wdv, dk[kk], aco[kk]);
                            agy[kk] = fmaf(wg, dk[kk], agy[kk]);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < CV; ++kk)
                            if (kk < c) acc[kk] = fmaf(w, vj[kk * TR_VS], acc[kk]);
                    }
                }
            }
            __syncwarp();  // the queue is refilled by the next block
        }
    }
    if (ok && CENTRED) {
        // 2d outputs per row: the partial layout uses a row width of 2d
        float* o = p.split > 1 ? p.part + (((size_t)ch * p.B + b) * p.nr + i) * (2 * d)
                               : p.out + ((size_t)b * p.nr + i) * p.ldo;
#pragma unroll
        for (int k = 0; k < TR_CD; ++k)
            if (k < d) {
                o[k] = aco[k];
                o[d + k] = agy[k];
            }
    } else if (ok) {
        float* o = p.split > 1 ? p.part + (((size_t)ch * p.B + b) * p.nr + i) * c
                               : p.out + ((size_t)b * p.nr + i) * p.ldo;
#pragma unroll
        for (int k = 0; k < CV; ++k)
            if (k < c) o[k] = acc[k];
    }
}

// out = sum over chunks of the partial sums, in chunk order.
__global__ void transport_merge_kernel(const float* part, long long count, int split, int c, int ldo, float* out) {
    const long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (e >= count) return;
    float s = 0.f;
    for (int ch = 0; ch < split; ++ch) s += part[(size_t)ch * count + e];
    out[(e / c) * ldo + e % c] = s;
}

__global__ void grad_finish_kernel(const float* P, const float* w, int B, int per_cloud, int d, float* g) {
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= (long long)B * per_cloud) return;
    const float wi = w ? w[i] : 1.f / (float)per_cloud;
    for (int k = 0; k < d; ++k) g[i * d + k] = 2.f * (wi * P[i * d + k] - g[i * d + k]);
}

cudaError_t launch_grad_finish(const float* P, const float* w, int B, int per_cloud, int d, float* g,
                               cudaStream_t st) {
    const long long count = (long long)B * per_cloud;
    if (count <= 0) return cudaSuccess;
    count_launches(1);
    grad_finish_kernel<<<(unsigned)((count + 255) / 256), 256, 0, st>>>(P, w, B, per_cloud, d, g);
    return cudaGetLastError();
}

using TrKernel = void (*)(TransportArgs);

// The kernel for d coordinates and c values per column (centred: the
// row-centred products, c = 1).
template <int CV, bool CENTRED = false>
static TrKernel tr_pick(int d) {
    if (d == 3) return transport_kernel<CV, 4, CENTRED, 3>;
    return tr_w(d) == 8 ? transport_kernel<CV, 8, CENTRED> : transport_kernel<CV, 4, CENTRED>;
}

static TrKernel tr_kernel(int d, int c, bool centred) {
    if (centred) return tr_pick<1, true>(d);
    if (c <= 1) return tr_pick<1>(d);
    if (c <= 4) return tr_pick<4>(d);
    if (c <= 16) return tr_pick<16>(d);
    return tr_pick<64>(d);
}

// CTAs of that kernel resident on one SM (4 when the device cannot say).
static int tr_resident(int d, int c, bool centred) {
    const TrKernel k = tr_kernel(d, c, centred);
    const size_t sm = tr_smem_bytes(d, centred ? 1 : c);
    int nb = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, TR_T, sm) != cudaSuccess || nb < 1) {
        (void)cudaGetLastError();
        return 4;
    }
    return nb;
}

size_t transport_plan(int B, int nr, int nc, int d, int c, bool centred, int sms, int* split, int* chunk) {
    // CTAs all do the same work, so the split is chosen for whole waves: the
    // fewest chunks, from one full wave of CTAs on, whose last wave is within
    // 2 % of the fullest any split gives.  A chunk keeps at least 8 column
    // tiles so that staging the rows stays a small part of its work.
    const long long blocks = (long long)B * ((nr + TR_T - 1) / TR_T);
    const long long cap = (long long)(sms > 0 ? sms : 152) * tr_resident(d, c, centred);
    const int tiles = (nc + TR_CT - 1) / TR_CT;
    const int smax = std::max(1, (tiles + 7) / 8);
    const int smin = (int)std::min<long long>(smax, std::max<long long>(1, (cap + blocks - 1) / blocks));
    int best_tpc = (tiles + smin - 1) / smin;
    double best = -1.0;
    for (int s = smin; s <= smax; ++s) {
        const int tpc = (tiles + s - 1) / s;
        if ((tiles + tpc - 1) / tpc != s) continue;  // the same chunks as a smaller s
        const long long g = blocks * s;
        const double fill = (double)g / (double)(((g + cap - 1) / cap) * cap);
        if (fill > best + 0.02) {
            best = fill;
            best_tpc = tpc;
        }
    }
    *chunk = best_tpc * TR_CT;
    *split = (nc + *chunk - 1) / *chunk;
    const size_t width = centred ? 2 * (size_t)d : (size_t)c;
    return *split > 1 ? (size_t)*split * B * nr * width : 0;
}

// Row-centred products (see CENTRED above): V holds g (c = 1, ldv = 1), out has
// ldo >= 2d; p.rc, p.rv are [B][nr][d].  The partial sums need split * B * nr * 2d floats.
cudaError_t launch_transport_centred(const TransportArgs& p, cudaStream_t st) {
    if (p.d < 1 || p.d > TR_CD || p.c != 1 || p.ldv != 1 || p.ldo < 2 * p.d || !p.rc || !p.rv || p.B < 1 ||
        p.nr < 1 || p.nc < 1 || p.split < 1 || p.chunk < 1 || (long long)p.split * p.chunk < p.nc ||
        (p.split > 1 && !p.part))
        return cudaErrorInvalidValue;
    const size_t sm = tr_smem_bytes(p.d, 1);
    dim3 grid(((p.nr + TR_T - 1) / TR_T) * p.split, p.B), block(TR_T);
    const TrKernel kern = tr_kernel(p.d, 1, true);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    count_launches(1);
    kern<<<grid, block, sm, st>>>(p);
    if (p.split > 1) {
        const long long count = (long long)p.B * p.nr * 2 * p.d;
        count_launches(1);
        transport_merge_kernel<<<(unsigned)((count + 255) / 256), 256, 0, st>>>(p.part, count, p.split, 2 * p.d,
                                                                                 p.ldo, p.out);
    }
    return cudaGetLastError();
}

cudaError_t launch_transport(const TransportArgs& p, cudaStream_t st) {
    if (p.d < 1 || p.d > TR_MAXD || p.c < 1 || p.c > TR_MAXC || p.B < 1 || p.nr < 1 || p.nc < 1 || p.split < 1 ||
        p.chunk < 1 || (long long)p.split * p.chunk < p.nc || (p.split > 1 && !p.part) || p.ldv < p.c ||
        p.ldo < p.c)
        return cudaErrorInvalidValue;
    const size_t sm = tr_smem_bytes(p.d, p.c);
    dim3 grid(((p.nr + TR_T - 1) / TR_T) * p.split, p.B), block(TR_T);
    const TrKernel kern = tr_kernel(p.d, p.c, false);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    count_launches(1);
    kern<<<grid, block, sm, st>>>(p);
    if (p.split > 1) {
        const long long count = (long long)p.B * p.nr * p.c;
        count_launches(1);
        transport_merge_kernel<<<(unsigned)((count + 255) / 256), 256, 0, st>>>(p.part, count, p.split, p.c, p.ldo,
                                                                                 p.out);
    }
    return cudaGetLastError();
}

}  // namespace sot
