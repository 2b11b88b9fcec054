// k_tc.cu -- Sinkhorn half-steps on the 5th-generation tensor cores
// (tcgen05, kind::f16) for d = 64.
//
// The half-step ("FlashSinkhorn", Methodologie 1-2) needs the dot products
// x_i . y_j of every (row, column) pair: a dense contraction over d = 64, so it
// runs on the tensor cores.  Single-pass fp16 (or tf32) products carry 11
// significant bits, which moves the gradient of the n = 70000 problem by
// ~3e-2 relative; fp32 accuracy comes from splitting every coordinate into
// an fp16 pair v = hi + lo and summing hi*hi + hi*lo + lo*hi (the lo*lo term
// is below fp32 rounding), all accumulated in fp32 in TMEM.
//
// Full half-step (tc_half_kernel), CTA layout (one CTA per SM; 320 threads):
//   warp 0      producer: bulk copies (TMA engine) of 128-column operand tiles
//               into a 4-stage shared-memory ring, plus the column biases
//               c_j = log2 w_j - Lam_j of each tile;
//   warp 1      MMA issuer (one thread) and TMEM owner (512 columns);
//   warps 2-9   two warpgroups, one per 128-row tile: tcgen05.ld of the fp32
//               accumulator, score = acc * 2 kappa / s^2 + c_j, ex2, row sums.
// The 256 rows of the CTA stay resident (row-stationary); every column tile
// is used by both row tiles (12 MMAs of 128 x 128 x 16 each) before its stage
// is released.  Accumulators are double-buffered per row tile so the MMAs of
// tile t+1 overlap the exponentials of tile t.  The screened half-step
// (tc_screen_kernel, below) keeps the roles with its own tile shapes.
//
// Operands live in HBM as images of the exact shared-memory layout (128-byte
// swizzle, K-major): per 128 points, 16 KB of hi parts then 16 KB of lo parts,
// so one 1-D bulk copy moves a whole tile.  Coordinates are scaled per cloud by
// a power of two s (max |s x| in (256, 512]) before the split; the epilogue
// divides by s^2.
//
// Every mbarrier wait is bounded (2 s of wall time, or as soon as another role
// gave up); a CTA that gives up poisons its rows with NaN, sets the device
// timeout bit, drains its own bulk copies, frees TMEM and returns.
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "tc.h"
#include "tc_ptx.cuh"

namespace sot {

constexpr int TC_D = 64;
constexpr int TC_M = 128;             // rows per row tile (MMA M)
constexpr int TC_ROWS = 2 * TC_M;     // rows per CTA
constexpr int TC_N = 128;             // columns per tile (MMA N)
constexpr int TC_S = 4;               // pipeline stages
constexpr int TC_THREADS = 320;
constexpr uint32_t TILE_BYTES = 16384;          // 128 x 64 fp16, one swizzled K-block
constexpr uint32_t OP_BYTES = 2 * TILE_BYTES;   // hi + lo
constexpr uint32_t OFF_A = 0;                           // [2 row tiles][hi, lo]
constexpr uint32_t OFF_B = OFF_A + 2 * OP_BYTES;        // [TC_S][hi, lo]
constexpr uint32_t OFF_BIAS = OFF_B + TC_S * OP_BYTES;  // [TC_S][TC_N] float
constexpr uint32_t OFF_BAR = OFF_BIAS + TC_S * TC_N * 4;
constexpr uint32_t NBAR = 18;
constexpr uint32_t OFF_MISC = OFF_BAR + 256;            // tmem slot, abort, nretry, last, pool count
constexpr uint32_t OFF_RED = OFF_MISC + 32;             // 32 floats (one per warp of a block reduction)
constexpr uint32_t OFF_RETRY = OFF_RED + 128;           // TC_ROWS ints
constexpr uint32_t TC_SMEM = OFF_RETRY + TC_ROWS * 4 + 1024;  // + alignment slack
constexpr uint64_t TC_WAIT_NS = 2000000000ull;

// barrier indices
__host__ __device__ constexpr int BAR_FULL(int s) { return s; }
__host__ __device__ constexpr int BAR_EMPTY(int s) { return TC_S + s; }
__host__ __device__ constexpr int BAR_ACCFULL(int r, int u) { return 2 * TC_S + 2 * r + u; }
__host__ __device__ constexpr int BAR_ACCEMPTY(int r, int u) { return 2 * TC_S + 4 + 2 * r + u; }
__host__ __device__ constexpr int BAR_A() { return 2 * TC_S + 8; }
__host__ __device__ constexpr int BAR_DRAIN() { return 2 * TC_S + 9; }  // every MMA of the CTA has completed
static_assert(BAR_DRAIN() + 1 == (int)NBAR, "barrier count");
static_assert(NBAR * 8 <= 256, "barriers fit the header");
static_assert(TC_SMEM <= 227 * 1024, "shared memory budget");

// Layout of the screened half-step: 256-column tiles (one 128 x 256 x 16 MMA
// per K step and row tile), a single 256-column TMEM accumulator per row tile.
constexpr int SC_N = 256;                                   // columns per screened tile (MMA N)
constexpr uint32_t SC_AT = TC_M * 32;                       // row-side constant block: 128 rows x 32 B (sw32)
constexpr uint32_t SC_BT = SC_N * 32;                       // bias block of a tile: 256 rows x 32 B (sw32)
constexpr int TC_MAXD = 1024;  // the screened half-step streams d in slices of 64 (K = 64 per image tile)

// Shared-memory layout of the screened half-step for NS slices of K = 64.
// Up to d = 256: the hi parts of both row tiles for every slice (resident),
// the row-side constant blocks, a ring of NST stages (one slice of one
// 256-column tile each, plus its bias block), then the header; wider d leaves
// room for fewer stages.  At d = 512 and 1024 (NS = 8, 16) the row tiles no
// longer fit: each stage also carries the slice of both row tiles, which are
// streamed again with every column tile.
template <int NS>
struct ScLayout {
    static constexpr bool STREAM = NS > 4;
    static constexpr uint32_t ST_B = STREAM ? 2 * TILE_BYTES : 0;  // a stage: [row tiles' slice], column tile's hi,
    static constexpr uint32_t ST_BIAS = ST_B + 2 * TILE_BYTES;     // then its bias block
    static constexpr uint32_t STAGE = ST_BIAS + SC_BT;
    static constexpr int NST = STREAM ? 2 : (NS == 1 ? 4 : (NS == 4 ? 2 : 3));
    static constexpr uint32_t OFF_A = 0;                                               // [2 row tiles][NS] hi
    static constexpr uint32_t OFF_AC = OFF_A + (STREAM ? 0u : 2u * NS * TILE_BYTES);  // [2 row tiles] constants
    static constexpr uint32_t OFF_B = OFF_AC + 2 * SC_AT;                              // [NST] stages
    static constexpr uint32_t OFF_HDR = OFF_B + NST * STAGE;  // header (as OFF_BAR.. of the full half-step)
    static constexpr uint32_t SMEM = OFF_HDR + (OFF_RETRY - OFF_BAR) + TC_ROWS * 4 + 1024;
};
static_assert(ScLayout<1>::OFF_B % 1024 == 0 && ScLayout<8>::OFF_B % 1024 == 0 && ScLayout<1>::STAGE % 1024 == 0 &&
                  ScLayout<8>::STAGE % 1024 == 0,
              "screened stage alignment");
static_assert(ScLayout<1>::SMEM <= 227 * 1024 && ScLayout<2>::SMEM <= 227 * 1024 &&
                  ScLayout<3>::SMEM <= 227 * 1024 && ScLayout<4>::SMEM <= 227 * 1024 &&
                  ScLayout<8>::SMEM <= 227 * 1024 && ScLayout<16>::SMEM <= 227 * 1024,
              "screened shared memory budget");
static_assert(ScLayout<4>::NST <= TC_S && ScLayout<1>::NST == TC_S && ScLayout<16>::NST <= TC_S, "stage barriers");

bool tc_supported(int d) { return d >= TC_D && d % TC_D == 0 && (d <= 256 || d == 512 || d == 1024); }
bool tc_half_supported(int d) { return tc_supported(d); }
int tc_max_d() { return TC_MAXD; }
int tc_rows_per_cta() { return TC_ROWS; }
int tc_cols_per_tile() { return SC_N; }  // column chunks are whole screened tiles
bool tc_apply_supported(int d) { return tc_supported(d); }
static inline int tc_slices(int d) { return d > TC_D ? d / TC_D : 1; }
// Automatic precision at d = 64 uses the tensor-core plan application.
bool tc_apply_default() { return true; }
int tc_apply_rows_per_cta() { return TC_ROWS; }

static inline int tc_tiles(int n) { return 2 * ((n + TC_ROWS - 1) / TC_ROWS); }

size_t tc_scratch_bytes(int B, int n, int m, int d) {
    const int tmax = tc_tiles(n) > tc_tiles(m) ? tc_tiles(n) : tc_tiles(m);
    return (size_t)B * (tc_tiles(n) + tc_tiles(m)) * tc_slices(d) * OP_BYTES + 256 + (size_t)B * 36 + 256 +
           (size_t)B * tmax * TC_N * sizeof(float) + 256 + (size_t)B * (tmax / 2) * SC_BT;
}

// ---- operand images -----------------------------------------------------------
__global__ void tc_maxabs_kernel(const float* xc, long long nx, const float* yc, long long ny, unsigned* maxbits) {
    const int b = blockIdx.y;
    const float* xb = xc + (size_t)b * nx;
    const float* yb = yc + (size_t)b * ny;
    float mx = 0.f;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < nx; e += (long long)gridDim.x * blockDim.x)
        mx = fmaxf(mx, fabsf(xb[e]));
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < ny; e += (long long)gridDim.x * blockDim.x)
        mx = fmaxf(mx, fabsf(yb[e]));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) atomicMax(maxbits + b, __float_as_uint(mx));
}

// scale[b] = 2^e with max|s x| in (256, 512]; exact power of two.
__device__ __forceinline__ float tc_scale_of(unsigned bits) {
    const float mx = __uint_as_float(bits);
    if (!(mx > 0.f) || !isfinite(mx)) return 1.f;
    int e;
    frexpf(mx, &e);  // mx = f * 2^e, f in [0.5, 1)
    return ldexpf(1.f, 9 - e);
}

// One thread per point (row of a 128-row tile): per slice of K = 64, 8 chunks
// of 8 fp16 for hi and lo (coordinates past d are zero).  Slice k of tile t
// of cloud b sits at ((b tiles + t) ns + k) OP_BYTES.
// nrm[b][0] / nrm[b][1] receive (as float bits, atomicMax) the largest norm of a
// point's hi part and of its exact residual v - hi, in scaled units: the
// screening margin of the hi * hi product is built from them.
__global__ void tc_image_kernel(const float* pc, int n, int d, int ns, int tiles, const unsigned* maxbits,
                                float* scale, unsigned char* img, unsigned* nrm, int nrm_stride) {
    const int b = blockIdx.y;
    const int tile = blockIdx.x;
    const int r = threadIdx.x;
    const int p = tile * TC_M + r;
    const float s = tc_scale_of(maxbits[b]);
    if (tile == 0 && r == 0) scale[b] = s;
    const float* src = pc + ((size_t)b * n + p) * d;
    float hh = 0.f, rr = 0.f;
    for (int c = 0; c < ns * (TC_D / 8); ++c) {
        const int sl = c / (TC_D / 8), cc = c % (TC_D / 8);
        unsigned char* hi = img + (((size_t)b * tiles + tile) * ns + sl) * OP_BYTES;
        unsigned char* lo = hi + TILE_BYTES;
        __align__(16) __half h[8], l[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int kk = 8 * c + k;
            const float v = (p < n && kk < d) ? src[kk] * s : 0.f;
            const __half hv = __float2half_rn(v);
            const float res = v - __half2float(hv);  // exact in fp32
            h[k] = hv;
            l[k] = __float2half_rn(res);
            hh = fmaf(__half2float(hv), __half2float(hv), hh);
            rr = fmaf(res, res, rr);
        }
        const uint32_t off = sw128_offset(r, 8 * cc);
        *reinterpret_cast<uint4*>(hi + off) = *reinterpret_cast<const uint4*>(h);
        *reinterpret_cast<uint4*>(lo + off) = *reinterpret_cast<const uint4*>(l);
    }
    if (nrm) {
        const float hn = warp_max(sqrtf(hh)), rn = warp_max(sqrtf(rr));
        if ((threadIdx.x & 31) == 0) {
            atomicMax(nrm + (size_t)b * nrm_stride, __float_as_uint(hn));
            atomicMax(nrm + (size_t)b * nrm_stride + 1, __float_as_uint(rn));
        }
    }
}

cudaError_t tc_prepare(TcPlan& plan, unsigned char* scratch, int B, int n, int m, int d, const float* xc,
                       const float* yc, cudaStream_t st) {
    if (!tc_supported(d)) return cudaErrorInvalidValue;
    plan.B = B; plan.n = n; plan.m = m; plan.d = d;
    plan.S = tc_slices(d);
    plan.tiles_x = tc_tiles(n);
    plan.tiles_y = tc_tiles(m);
    uintptr_t base = ((uintptr_t)scratch + 255) & ~(uintptr_t)255;
    plan.xop = reinterpret_cast<unsigned char*>(base);
    plan.yop = plan.xop + (size_t)B * plan.tiles_x * plan.S * OP_BYTES;
    unsigned* maxbits = reinterpret_cast<unsigned*>(plan.yop + (size_t)B * plan.tiles_y * plan.S * OP_BYTES);
    plan.scale = reinterpret_cast<float*>(maxbits + B);
    plan.nrm = reinterpret_cast<unsigned*>(plan.scale + B);
    plan.cmax = plan.nrm + 4 * B;
    plan.bias = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(plan.cmax + 3 * B) + 255) & ~(uintptr_t)255);
    {
        const int tmax = plan.tiles_x > plan.tiles_y ? plan.tiles_x : plan.tiles_y;
        plan.bimg = reinterpret_cast<unsigned char*>(
            (reinterpret_cast<uintptr_t>(plan.bias + (size_t)B * tmax * TC_N) + 255) & ~(uintptr_t)255);
    }
    cudaError_t e = cudaMemsetAsync(maxbits, 0, sizeof(unsigned) * B * 9, st);  // maxbits, scale, nrm, cmax
    if (e != cudaSuccess) return e;
    count_launches(1);
    tc_maxabs_kernel<<<dim3(64, B), 256, 0, st>>>(xc, (long long)n * d, yc, (long long)m * d, maxbits);
    count_launches(1);
    tc_image_kernel<<<dim3(plan.tiles_x, B), TC_M, 0, st>>>(xc, n, d, plan.S, plan.tiles_x, maxbits, plan.scale,
                                                            plan.xop, plan.nrm, 4);
    count_launches(1);
    tc_image_kernel<<<dim3(plan.tiles_y, B), TC_M, 0, st>>>(yc, m, d, plan.S, plan.tiles_y, maxbits, plan.scale,
                                                            plan.yop, plan.nrm + 2, 4);
    return cudaGetLastError();
}

// ---- shared machinery of the tensor-core kernels ----------------------------------
struct TcOps {
    const unsigned char* aimg;  // row-side image
    const unsigned char* bimg;  // column-side image
    const float* scale;
    const float* bias;          // [B][tiles_c * TC_N] column biases c_j, -inf past the last column
    const unsigned char* bias_img;  // [B][tiles_c] 16 KB tiles: fp16 bias parts (screened half-step)
    int tiles_r, tiles_c;
    int S;                          // slices of K = 64 per image tile
    int hold_tile;                  // testing hook: the producer issues no copy from this column tile of its
                                    // chunk on (-1: off), so the waits on it run out
    unsigned long long wait_ns;     // limit of every bounded wait
};

// Host-side settings every tensor-core launch copies into TcOps.
static std::atomic<int> g_hold_tile{-1};
static std::atomic<int> g_hold_after{0};  // launches left alone before the hook applies
static std::atomic<unsigned long long> g_wait_ns{TC_WAIT_NS};

void tc_set_test_hold(int tile, int after, unsigned long long wait_ns) {
    g_hold_after.store(after > 0 ? after : 0);
    g_hold_tile.store(tile < 0 ? -1 : tile);
    g_wait_ns.store(wait_ns > 0 ? wait_ns : TC_WAIT_NS);
}

static void tc_fill_waits(TcOps& ops) {
    ops.hold_tile = g_hold_tile.load();
    ops.wait_ns = g_wait_ns.load();
    if (ops.hold_tile >= 0 && g_hold_after.load() > 0 && g_hold_after.fetch_sub(1) > 0) ops.hold_tile = -1;
}

// Column biases of one half-step, c_j = log2 w_j - state_j, padded with -inf
// to whole tiles: the producer moves a tile's biases with one bulk copy.
__global__ void tc_bias_kernel(const float* cw, const float* cst, int nc, int nc_pad, float* bias) {
    const int b = blockIdx.y;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nc_pad; j += gridDim.x * blockDim.x)
        bias[(size_t)b * nc_pad + j] = (j < nc) ? cw[(size_t)b * nc + j] - cst[(size_t)b * nc + j] : -INFINITY;
}

static cudaError_t launch_tc_bias(const TcPlan& plan, const HalfArgs& p, int tiles_c, cudaStream_t st) {
    const int nc_pad = tiles_c * TC_N;
    const int blocks = (nc_pad + 255) / 256 < 1024 ? (nc_pad + 255) / 256 : 1024;
    count_launches(1);
    tc_bias_kernel<<<dim3(blocks, p.B), 256, 0, st>>>(p.cw2, p.cstate, p.nc, nc_pad, plan.bias);
    return cudaGetLastError();
}

// ---- column biases of the screened half-step, added by the tensor cores --------
// The screened half-step lets the MMA add the column bias c_j to the hi * hi
// products: one more K = 16 step multiplies a row-side constant block
// (2^E, 2^(E-11), 2^(E-22), 0, ...) by a column-side block (b1, b2, b3, 0, ...)
// with c_j / tk = 2^E b1 + 2^(E-11) b2 + 2^(E-22) b3 (three fp16 parts, ~33
// significant bits; tk = 2 kappa / s^2 turns accumulator units into log2
// units).  Every product is exact; the accumulator then holds score / tk.
// E is chosen per cloud from max_j |c_j| so that |b1| < 2^15; a cloud that
// would need E > 15 cannot be screened (its rows take the exact full LSE).

// E of one cloud from max |c_j| (float bits) and the coordinate scale; both
// the bias image and the row-side constants use this same computation.
__device__ __forceinline__ int tc_bias_exp(unsigned cmax_bits, float s, float two_kappa) {
    const float mb = __uint_as_float(cmax_bits) * (s * s / two_kappa);
    if (!(mb > 0.f)) return -2;
    if (!isfinite(mb)) return 99;
    const int e = ilogbf(mb) - 14;
    return e < -2 ? -2 : e;
}

// max_j |c_j| per cloud into cmax[2B + b] (float bits).  Warp maxima go to
// cmax[b] with atomicMax (non-negative floats order as their bits); the last
// block of the cloud moves the result and clears the running slots.
__global__ void tc_cmax_kernel(const float* cw, const float* cst, int nc, unsigned* cmax) {
    const int b = blockIdx.y, B = gridDim.y;
    float mx = 0.f;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nc; j += gridDim.x * blockDim.x)
        mx = fmaxf(mx, fabsf(cw[(size_t)b * nc + j] - cst[(size_t)b * nc + j]));
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) atomicMax(cmax + b, __float_as_uint(mx));
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(cmax + B + b, 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            cmax[2 * B + b] = atomicExch(cmax + b, 0u);
            cmax[B + b] = 0u;
        }
    }
}

// Column side of the bias step: per column j, the parts (b1, b2, b3) as fp16
// K-elements 0..2 (3..15 zero) of row j % 256 of the 32-byte-swizzled K-major
// block of its 256-column tile (8 KB).  Columns past nc get b1 = -inf, so
// their scores are -inf.
__global__ void tc_bias_image_kernel(const float* cw, const float* cst, int nc, int nc_pad, const float* scale,
                                     float two_kappa, const unsigned* cmax, unsigned char* img) {
    const int b = blockIdx.y, B = gridDim.y;
    const float s = scale[b];
    const float inv_tk = s * s / two_kappa;
    const int E = tc_bias_exp(cmax[2 * B + b], s, two_kappa);
    const float sc1 = ldexpf(1.f, E > 15 ? 0 : -E);
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nc_pad; j += gridDim.x * blockDim.x) {
        __half h0 = __float2half_rn(0.f), h1 = h0, h2 = h0;
        if (j < nc) {
            const float v = (cw[(size_t)b * nc + j] - cst[(size_t)b * nc + j]) * inv_tk * sc1;
            if (E <= 15 && isfinite(v)) {
                h0 = __float2half_rn(v);
                const float r1 = (v - __half2float(h0)) * 2048.f;  // exact: the bits of v below h0
                h1 = __float2half_rn(r1);
                const float r2 = (r1 - __half2float(h1)) * 2048.f;
                h2 = __float2half_rn(r2);
            } else if (E <= 15) {
                h0 = __float2half_rn(v);  // a NaN bias stays NaN: the pair is never kept
            }
        } else {
            h0 = __float2half_rn(-INFINITY);
        }
        unsigned char* tile = img + ((size_t)b * (nc_pad / SC_N) + j / SC_N) * SC_BT;
        const int jr = j % SC_N;
        *reinterpret_cast<uint4*>(tile + sw32_offset(jr, 0)) =
            make_uint4((unsigned)__half_as_ushort(h0) | ((unsigned)__half_as_ushort(h1) << 16),
                       (unsigned)__half_as_ushort(h2), 0u, 0u);
        *reinterpret_cast<uint4*>(tile + sw32_offset(jr, 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

static cudaError_t launch_tc_bias_image(const TcPlan& plan, const HalfArgs& p, int tiles_c, cudaStream_t st) {
    const int nc_pad = tiles_c * TC_N;
    int blocks = (p.nc + 255) / 256 < 1024 ? (p.nc + 255) / 256 : 1024;
    if (blocks < 1) blocks = 1;
    count_launches(1);
    tc_cmax_kernel<<<dim3(blocks, p.B), 256, 0, st>>>(p.cw2, p.cstate, p.nc, plan.cmax);
    blocks = (nc_pad + 255) / 256 < 1024 ? (nc_pad + 255) / 256 : 1024;
    count_launches(1);
    tc_bias_image_kernel<<<dim3(blocks, p.B), 256, 0, st>>>(p.cw2, p.cstate, p.nc, nc_pad, plan.scale, p.two_kappa,
                                                            plan.cmax, plan.bimg);
    return cudaGetLastError();
}

// The header (barriers, misc words, reduction scratch, retry list) sits at
// `hdr`: after the operand buffers, whose layout differs between kernels.
struct TcSmem {
    uint32_t sbase;       // 1024-aligned shared address of the layout
    unsigned char* sm;    // generic pointer to the same place
    uint32_t hdr;         // offset of the header
    __device__ uint32_t bar(int i) const { return sbase + hdr + 8u * (uint32_t)i; }
    __device__ float* bias() const { return reinterpret_cast<float*>(sm + OFF_BIAS); }
    __device__ uint32_t misc_addr() const { return sbase + hdr + (OFF_MISC - OFF_BAR); }
    __device__ int* misc() const { return reinterpret_cast<int*>(sm + hdr + (OFF_MISC - OFF_BAR)); }  // tmem, abort, nretry, last, pool
    __device__ volatile int* abort() const { return misc() + 1; }
    __device__ float* red() const { return reinterpret_cast<float*>(sm + hdr + (OFF_RED - OFF_BAR)); }
    __device__ int* retry() const { return reinterpret_cast<int*>(sm + hdr + (OFF_RETRY - OFF_BAR)); }
};

__device__ __forceinline__ TcSmem tc_smem(unsigned char* raw_ptr, uint32_t hdr = OFF_BAR) {
    TcSmem S;
    const uint32_t raw = smem_u32(raw_ptr);
    S.sbase = (raw + 1023u) & ~1023u;
    S.sm = raw_ptr + (S.sbase - raw);
    S.hdr = hdr;
    return S;
}

// Barriers, TMEM allocation (warp 1, 512 columns); returns the TMEM base address.
// `empty_count`: arrivals that free a stage (the MMA commit, plus one per
// epilogue warp when the epilogue reads the stage's biases).
// `accempty_count`: epilogue warps that read (and free) one accumulator buffer.
// `empty_count_hi`: when nonzero, the arrivals that free stages TC_S / 2 ..
// (the bias slots of the sliced full half-step).
__device__ __forceinline__ uint32_t tc_setup(const TcSmem& S, int warp, uint32_t empty_count = 1 + 8,
                                             uint32_t accempty_count = 4, uint32_t empty_count_hi = 0) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_S; ++s) {
            mbar_init(S.bar(BAR_FULL(s)), 1);
            mbar_init(S.bar(BAR_EMPTY(s)), (empty_count_hi && s >= TC_S / 2) ? empty_count_hi : empty_count);
        }
        for (int r = 0; r < 2; ++r)
            for (int u = 0; u < 2; ++u) {
                mbar_init(S.bar(BAR_ACCFULL(r, u)), 1);
                mbar_init(S.bar(BAR_ACCEMPTY(r, u)), accempty_count);
            }
        mbar_init(S.bar(BAR_A()), 1);
        mbar_init(S.bar(BAR_DRAIN()), 1);
        S.misc()[1] = 0;
        S.misc()[2] = 0;
        S.misc()[4] = 0;
        S.misc()[5] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(S.misc_addr(), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return (uint32_t)S.misc()[0];
}

// Never leave a bulk copy in flight into this CTA's shared memory: waits
// (bounded, and not cut short by the abort flag) for the last nst stages
// issued (a ring of nst stages) and for the row tiles.
__device__ __forceinline__ void tc_producer_drain(const TcSmem& S, int issued, uint64_t wait_ns, int nst = TC_S) {
    if ((threadIdx.x & 31) == 0) {
        int dummy = 0;
        for (int lt = (issued > nst ? issued - nst : 0); lt < issued; ++lt)
            mbar_wait_bounded(S.bar(BAR_FULL(lt % nst)), (uint32_t)(lt / nst) & 1u, (volatile int*)&dummy,
                              wait_ns);
        mbar_wait_bounded(S.bar(BAR_A()), 0u, (volatile int*)&dummy, wait_ns);
    }
    __syncwarp();
}

// Never leave an MMA in flight when the CTA frees TMEM and exits: the MMA
// thread commits everything it issued to the drain barrier and waits for it
// (bounded, and not cut short by the abort flag).  On the normal path the
// MMAs have completed by then or are about to.
__device__ __forceinline__ void tc_mma_drain(const TcSmem& S, bool issued_any, uint64_t wait_ns) {
    if (!issued_any) return;
    int dummy = 0;
    tc_commit(S.bar(BAR_DRAIN()));
    mbar_wait_bounded(S.bar(BAR_DRAIN()), 0u, (volatile int*)&dummy, wait_ns);
}

// Producer warp (lane 0 issues): the CTA's two row tiles once, then the
// column tiles of the chunk through the TC_S-stage ring, each with its 128
// fp32 column biases, all by bulk copies completing on the stage's barrier.
__device__ void tc_producer(const TcSmem& S, const TcOps& ops, int b, int rb, int t0, int nt) {
    const int lane = threadIdx.x & 31;
    volatile int* abort = S.abort();
    int issued = 0;
    if (lane == 0) {
        const unsigned char* a0 = ops.aimg + ((size_t)b * ops.tiles_r + 2 * rb) * OP_BYTES;
        mbar_arrive_expect_tx(S.bar(BAR_A()), 2 * OP_BYTES);
        bulk_g2s(S.sbase + OFF_A, a0, 2 * OP_BYTES, S.bar(BAR_A()));
    }
    const unsigned char* bimg = ops.bimg + (size_t)b * ops.tiles_c * OP_BYTES;
    const float* gbias = ops.bias + (size_t)b * ops.tiles_c * TC_N;
    for (int lt = 0; lt < nt; ++lt) {
        if (lt == ops.hold_tile) break;
        const int st = lt % TC_S;
        const uint32_t ph = (uint32_t)(lt / TC_S) & 1u;
        if (!mbar_wait_bounded(S.bar(BAR_EMPTY(st)), ph ^ 1u, abort, ops.wait_ns)) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(S.bar(BAR_FULL(st)), OP_BYTES + TC_N * 4);
            bulk_g2s(S.sbase + OFF_B + (uint32_t)st * OP_BYTES, bimg + (size_t)(t0 + lt) * OP_BYTES, OP_BYTES,
                     S.bar(BAR_FULL(st)));
            bulk_g2s(S.sbase + OFF_BIAS + (uint32_t)st * TC_N * 4, gbias + (size_t)(t0 + lt) * TC_N, TC_N * 4,
                     S.bar(BAR_FULL(st)));
        }
        issued = lt + 1;
    }
    tc_producer_drain(S, issued, ops.wait_ns);
}

// MMA warp (one thread): per column tile and row tile, 12 MMAs of
// 128 x 128 x 16 -- lo*hi and hi*lo first, then hi*hi -- into the row tile's
// TMEM buffer (lt & 1); commits signal the epilogue and free the stage.
__device__ void tc_mma(const TcSmem& S, uint32_t tmem, int nt, uint64_t wait_ns) {
    if ((threadIdx.x & 31) == 0) {
        volatile int* abort = S.abort();
        bool ok = mbar_wait_bounded(S.bar(BAR_A()), 0u, abort, wait_ns);
        bool issued_any = false;
        const uint32_t idesc = f16_idesc(TC_M, TC_N);
        for (int lt = 0; ok && lt < nt; ++lt) {
            const int st = lt % TC_S;
            const uint32_t ph = (uint32_t)(lt / TC_S) & 1u;
            const int u = lt & 1;
            const uint32_t pu = (uint32_t)(lt >> 1) & 1u;
            if (!mbar_wait_bounded(S.bar(BAR_FULL(st)), ph, abort, wait_ns)) break;
            for (int r = 0; r < 2 && ok; ++r) {
                if (!mbar_wait_bounded(S.bar(BAR_ACCEMPTY(r, u)), pu ^ 1u, abort, wait_ns)) { ok = false; break; }
                tc_fence_after();
                issued_any = true;
                const uint32_t d = tmem + (uint32_t)((2 * r + u) * TC_N);
                const uint32_t ahi = S.sbase + OFF_A + (uint32_t)r * OP_BYTES, alo = ahi + TILE_BYTES;
                const uint32_t bhi = S.sbase + OFF_B + (uint32_t)st * OP_BYTES, blo = bhi + TILE_BYTES;
#pragma unroll
                for (int k = 0; k < TC_D / 16; ++k) {
                    const uint32_t ko = 32u * (uint32_t)k;
                    tc_mma_f16(d, sw128_desc(ahi + ko), sw128_desc(blo + ko), idesc, k > 0 ? 1u : 0u);
                    tc_mma_f16(d, sw128_desc(alo + ko), sw128_desc(bhi + ko), idesc, 1u);
                }
#pragma unroll
                for (int k = 0; k < TC_D / 16; ++k) {
                    const uint32_t ko = 32u * (uint32_t)k;
                    tc_mma_f16(d, sw128_desc(ahi + ko), sw128_desc(bhi + ko), idesc, 1u);
                }
                tc_commit(S.bar(BAR_ACCFULL(r, u)));
            }
            if (!ok) break;
            tc_commit(S.bar(BAR_EMPTY(st)));
        }
        tc_mma_drain(S, issued_any, wait_ns);
    }
    __syncwarp();
}

// ---- the full half-step at d = 128 ... 1024 (ns slices of K = 64) ----------
// The row tiles' hi and lo parts (64 KB a slice) no longer stay resident:
// each of two operand stages (96 KB) carries one slice of both row tiles and
// of the column tile, hi and lo, and the accumulator gathers the slices.  The
// column biases go to two slots of their own (one per accumulator buffer),
// loaded with the tile's first slice and freed by the epilogue.
constexpr int TCS_ST = 2;                      // operand stages
constexpr uint32_t TCS_STAGE = 3 * OP_BYTES;   // [row tile 0][row tile 1][column tile], hi + lo each
static_assert(TCS_ST * TCS_STAGE <= OFF_BIAS && TCS_STAGE % 1024 == 0, "sliced operand stages");
static_assert(TCS_ST == TC_S / 2, "bias slots use the upper stage barriers");
__host__ __device__ constexpr int BAR_BFULL(int u) { return BAR_FULL(TCS_ST + u); }
__host__ __device__ constexpr int BAR_BEMPTY(int u) { return BAR_EMPTY(TCS_ST + u); }

__device__ void tc_producer_sl(const TcSmem& S, const TcOps& ops, int b, int rb, int t0, int nt, int ns) {
    const int lane = threadIdx.x & 31;
    volatile int* abort = S.abort();
    int issued = 0, bissued = 0;
    if (lane == 0) mbar_arrive(S.bar(BAR_A()));  // nothing resident: the wait on the row tiles passes at once
    const float* gbias = ops.bias + (size_t)b * ops.tiles_c * TC_N;
    bool ok = true;
    for (int lt = 0; ok && lt < nt; ++lt) {
        if (lt == ops.hold_tile) break;
        const int u = lt & 1;
        if (!mbar_wait_bounded(S.bar(BAR_BEMPTY(u)), ((uint32_t)(lt >> 1) & 1u) ^ 1u, abort, ops.wait_ns)) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(S.bar(BAR_BFULL(u)), TC_N * 4);
            bulk_g2s(S.sbase + OFF_BIAS + (uint32_t)u * TC_N * 4, gbias + (size_t)(t0 + lt) * TC_N, TC_N * 4,
                     S.bar(BAR_BFULL(u)));
        }
        bissued = lt + 1;
        for (int k = 0; k < ns; ++k) {
            const int it = lt * ns + k, st = it % TCS_ST;
            const uint32_t ph = (uint32_t)(it / TCS_ST) & 1u;
            if (!mbar_wait_bounded(S.bar(BAR_EMPTY(st)), ph ^ 1u, abort, ops.wait_ns)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = S.sbase + (uint32_t)st * TCS_STAGE;
                mbar_arrive_expect_tx(S.bar(BAR_FULL(st)), TCS_STAGE);
                for (int r = 0; r < 2; ++r)
                    bulk_g2s(dst + (uint32_t)r * OP_BYTES,
                             ops.aimg + (((size_t)b * ops.tiles_r + 2 * rb + r) * ns + k) * OP_BYTES, OP_BYTES,
                             S.bar(BAR_FULL(st)));
                bulk_g2s(dst + 2 * OP_BYTES, ops.bimg + (((size_t)b * ops.tiles_c + t0 + lt) * ns + k) * OP_BYTES,
                         OP_BYTES, S.bar(BAR_FULL(st)));
            }
            issued = it + 1;
        }
    }
    // never leave a copy in flight: the last stages and bias slots issued
    if (lane == 0) {
        int dummy = 0;
        for (int it = (issued > TCS_ST ? issued - TCS_ST : 0); it < issued; ++it)
            mbar_wait_bounded(S.bar(BAR_FULL(it % TCS_ST)), (uint32_t)(it / TCS_ST) & 1u, (volatile int*)&dummy,
                              ops.wait_ns);
        for (int lt = (bissued > 2 ? bissued - 2 : 0); lt < bissued; ++lt)
            mbar_wait_bounded(S.bar(BAR_BFULL(lt & 1)), (uint32_t)(lt >> 1) & 1u, (volatile int*)&dummy,
                              ops.wait_ns);
        mbar_wait_bounded(S.bar(BAR_A()), 0u, (volatile int*)&dummy, ops.wait_ns);
    }
    __syncwarp();
}

// Per column tile, row tile and slice: 4 lo*hi + 4 hi*lo, then 4 hi*hi
// 128 x 128 x 16 MMAs into the row tile's buffer (lt & 1), committed after
// the last slice; each slice's stage is freed by its own commit.
__device__ void tc_mma_sl(const TcSmem& S, uint32_t tmem, int nt, int ns, uint64_t wait_ns) {
    if ((threadIdx.x & 31) == 0) {
        volatile int* abort = S.abort();
        bool ok = mbar_wait_bounded(S.bar(BAR_A()), 0u, abort, wait_ns);
        bool issued_any = false;
        const uint32_t idesc = f16_idesc(TC_M, TC_N);
        for (int lt = 0; ok && lt < nt; ++lt) {
            const int u = lt & 1;
            const uint32_t pu = (uint32_t)(lt >> 1) & 1u;
            for (int k = 0; ok && k < ns; ++k) {
                const int it = lt * ns + k, st = it % TCS_ST;
                const uint32_t ph = (uint32_t)(it / TCS_ST) & 1u;
                if (!mbar_wait_bounded(S.bar(BAR_FULL(st)), ph, abort, wait_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t base = S.sbase + (uint32_t)st * TCS_STAGE;
                for (int r = 0; r < 2 && ok; ++r) {
                    if (k == 0) {
                        if (!mbar_wait_bounded(S.bar(BAR_ACCEMPTY(r, u)), pu ^ 1u, abort, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    issued_any = true;
                    const uint32_t d = tmem + (uint32_t)((2 * r + u) * TC_N);
                    const uint32_t ahi = base + (uint32_t)r * OP_BYTES, alo = ahi + TILE_BYTES;
                    const uint32_t bhi = base + 2 * OP_BYTES, blo = bhi + TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_D / 16; ++kk) {
                        const uint32_t ko = 32u * (uint32_t)kk;
                        tc_mma_f16(d, sw128_desc(ahi + ko), sw128_desc(blo + ko), idesc, (k > 0 || kk > 0) ? 1u : 0u);
                        tc_mma_f16(d, sw128_desc(alo + ko), sw128_desc(bhi + ko), idesc, 1u);
                    }
#pragma unroll
                    for (int kk = 0; kk < TC_D / 16; ++kk) {
                        const uint32_t ko = 32u * (uint32_t)kk;
                        tc_mma_f16(d, sw128_desc(ahi + ko), sw128_desc(bhi + ko), idesc, 1u);
                    }
                    if (k == ns - 1) tc_commit(S.bar(BAR_ACCFULL(r, u)));
                }
                if (!ok) break;
                tc_commit(S.bar(BAR_EMPTY(st)));
            }
        }
        tc_mma_drain(S, issued_any, wait_ns);
    }
    __syncwarp();
}

// After an epilogue warp has consumed tile lt: release its TMEM buffer and its stage.
__device__ __forceinline__ void tc_release(const TcSmem& S, int wg, int lt) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        mbar_arrive(S.bar(BAR_ACCEMPTY(wg, lt & 1)));
        mbar_arrive(S.bar(BAR_EMPTY(lt % TC_S)));
    }
}

// Exact two-pass LSE of one row over all columns, by the whole CTA (the
// fallback for rows whose fast path could not give the value): fp32 dot
// products of the centred coordinates, y read as float4.  DC = TC_D keeps
// the row in registers; DC = 0 takes any d (a multiple of 4) and reads the
// row per column (L1).  The d = 64 form is kept as it is: the register
// allocation of the kernels that inline it depends on it.
template <int NT, int DC>
__device__ float tc_row_full(const float* rows, const float* cols, const float* cw, const float* cst, int nc, int d,
                             int row, float tk, float* red) {
    const float4* xr = reinterpret_cast<const float4*>(rows + (size_t)row * d);
    float4 xv[DC > 0 ? DC / 4 : 1];
#pragma unroll
    for (int q = 0; q < (DC > 0 ? DC / 4 : 0); ++q) xv[q] = xr[q];
    auto score = [&](int j) {
        const float4* y = reinterpret_cast<const float4*>(cols + (size_t)j * d);
        float a0 = 0.f, a1 = 0.f;
        if (DC > 0) {
#pragma unroll
            for (int q = 0; q < (DC > 0 ? DC / 4 : 0); ++q) {
                const float4 v = __ldg(y + q);
                a0 = fmaf(xv[q].x, v.x, a0);
                a1 = fmaf(xv[q].y, v.y, a1);
                a0 = fmaf(xv[q].z, v.z, a0);
                a1 = fmaf(xv[q].w, v.w, a1);
            }
        } else {
#pragma unroll 4
            for (int q = 0; q < d / 4; ++q) {
                const float4 x4 = __ldg(xr + q), v = __ldg(y + q);
                a0 = fmaf(x4.x, v.x, a0);
                a1 = fmaf(x4.y, v.y, a1);
                a0 = fmaf(x4.z, v.z, a0);
                a1 = fmaf(x4.w, v.w, a1);
            }
        }
        return fmaf(tk, a0 + a1, cw[j] - cst[j]);
    };
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < nc; j += NT) mx = fmaxf(mx, score(j));
    mx = block_max<NT>(mx, red);
    if (mx == -INFINITY) return -INFINITY;
    float sm = 0.f;
    for (int j = threadIdx.x; j < nc; j += NT) sm += ex2f(score(j) - mx);
    sm = block_sum<NT>(sm, red);
    return mx + log2f(sm);
}

// Common end of the half-step kernels, run by the CTA that holds the final
// row values: rows queued in the retry list get the exact two-pass row LSE
// (whole CTA), then the marginal-error partial and the bound for the next
// half-step are formed from the new row values.
template <int NT, int DC>
__device__ void tc_tail(const HalfArgs& p, const TcSmem& S, bool erow, int row, float old, int b, int rb,
                        size_t rbase, const float* cw, const float* cst) {
    int* misc = S.misc();
    float* red = S.red();
    const int* retry = S.retry();
    const int lane = threadIdx.x & 31;
    __syncthreads();
    const int nretry = misc[2];
    const float* rows_fp32 = p.rpack + (size_t)b * p.nr * p.d;
    const float* cols_fp32 = p.cpack + (size_t)b * p.nc * p.d;
    for (int k = 0; k < nretry; ++k) {
        const int r = retry[k];
        const float v = tc_row_full<NT, DC>(rows_fp32, cols_fp32, cw, cst, p.nc, p.d, r, p.two_kappa, red);
        if (threadIdx.x == 0) {
            p.rstate_out[rbase + r] = v;
            atomicOr(p.status, SOT_DEV_RETRY_ROWS);
        }
    }
    if (p.errpart || p.lo_out) {
        __syncthreads();
        float e = 0.f, lo = INFINITY;
        if (erow) {
            const float nv = p.rstate_out[rbase + row];
            const float w = p.rweight ? p.rweight[rbase + row] : 1.f / (float)p.nr;
            e = w * fabsf(ex2f(nv - old) - 1.f);
            lo = old - nv;
        }
        if (p.errpart) {
            e = block_sum<NT>(e, red);
            if (threadIdx.x == 0) p.errpart[b * p.rowtiles + rb] = e;
        }
        if (p.lo_out) {
            lo = warp_min(lo);
            if (lane == 0 && lo < INFINITY) atomicMin(p.lo_out + b, ord_encode(lo));
        }
    }
}

// ---- the half-step ------------------------------------------------------------------
// SL: d > 64, the operands stream in slices (tc_producer_sl / tc_mma_sl).
template <bool SL>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_half_kernel(HalfArgs p, TcOps ops) {
    if (p.stop_flag && *(volatile const int*)p.stop_flag) return;
    // (after a screened half-step on probation: only the row blocks it left)
    if (p.redo && !p.redo[(size_t)blockIdx.y * p.rowtiles + blockIdx.x / p.split]) return;
    extern __shared__ unsigned char smem_raw[];
    const TcSmem S = tc_smem(smem_raw);
    int* misc = S.misc();
    volatile int* abort = S.abort();
    float* red = S.red();
    int* retry = S.retry();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int rb = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rb * TC_ROWS;
    const int c_begin = ch * p.chunk;
    const int c_end = min(p.nc, c_begin + p.chunk);
    const int t0 = c_begin / TC_N;
    const int nt = (c_end - c_begin + TC_N - 1) / TC_N;
    const float* cw = p.cw2 + (size_t)b * p.nc;
    const float* cst = p.cstate + (size_t)b * p.nc;
    const size_t rbase = (size_t)b * p.nr;
    const float sc = ops.scale[b];
    const float tk = p.two_kappa / (sc * sc);

    if (p.lo_reset && blockIdx.x == 0 && blockIdx.y == 0)
        for (int k = threadIdx.x; k < p.B; k += TC_THREADS) p.lo_reset[k] = SOT_ORD_EMPTY;
    // sliced: operand stages freed by the MMA commit alone, bias slots by the 8 epilogue warps
    const uint32_t tmem = SL ? tc_setup(S, warp, 1, 4, 8) : tc_setup(S, warp);

    float m = 0.f, s = 0.f;  // epilogue row state
    const int wg = (warp - 2) >> 2;  // row tile of this epilogue warp
    const int q4 = warp & 3;         // TMEM lane quarter this warp may access
    const int row = row0 + wg * TC_M + q4 * 32 + lane;
    const bool erow = (warp >= 2) && row < p.nr;
    const float old = (erow && p.rstate_in) ? p.rstate_in[rbase + row] : 0.f;

    if (warp == 0) {
        if (SL) tc_producer_sl(S, ops, b, rb, t0, nt, ops.S);
        else tc_producer(S, ops, b, rb, t0, nt);
    } else if (warp == 1) {
        if (SL) tc_mma_sl(S, tmem, nt, ops.S, ops.wait_ns);
        else tc_mma(S, tmem, nt, ops.wait_ns);
    } else {
        // ---------------- epilogue: exponentials and row sums ----------------
        m = erow ? stabiliser(p.cold, p.lo_in, b, old) : INFINITY;
        s = 0.f;
        const float2 tk2 = make_float2(tk, tk);
        const float* bias = S.bias();
        for (int lt = 0; lt < nt; ++lt) {
            const int st = lt % TC_S;
            const uint32_t ph = (uint32_t)(lt / TC_S) & 1u;
            const int u = lt & 1;
            const uint32_t pu = (uint32_t)(lt >> 1) & 1u;
            // the tile's biases: in its stage, or (sliced) in bias slot u
            if (!mbar_wait_bounded(S.bar(SL ? BAR_BFULL(u) : BAR_FULL(st)), SL ? pu : ph, abort, ops.wait_ns)) break;
            if (!mbar_wait_bounded(S.bar(BAR_ACCFULL(wg, u)), pu, abort, ops.wait_ns)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)((2 * wg + u) * TC_N);
            const float* cb = bias + (SL ? u : st) * TC_N;
            const float2 nm2 = make_float2(-m, -m);
            float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int q = 0; q < TC_N / 32; ++q) {
                float v[32];
                tmem_ld32(tb + 32u * (uint32_t)q, v);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(cb + 32 * q + j);
                    float2 t = ffma2(make_float2(v[j], v[j + 1]), tk2, make_float2(c4.x, c4.y));
                    t = fadd2(t, nm2);
                    acc2 = fadd2(acc2, make_float2(ex2f(t.x), ex2f(t.y)));
                    t = ffma2(make_float2(v[j + 2], v[j + 3]), tk2, make_float2(c4.z, c4.w));
                    t = fadd2(t, nm2);
                    acc2 = fadd2(acc2, make_float2(ex2f(t.x), ex2f(t.y)));
                }
            }
            float ts = acc2.x + acc2.y;
            const bool ovf = !(ts < SOT_TILE_SUM_MAX);
            if (__any_sync(0xffffffffu, ovf)) {
                // warp-uniform slow path: re-stabilise overflowing rows on the tile maximum
                float mt = -INFINITY;
#pragma unroll 1
                for (int q = 0; q < TC_N / 32; ++q) {
                    float v[32];
                    tmem_ld32(tb + 32u * (uint32_t)q, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) mt = fmaxf(mt, fmaf(v[j], tk, cb[32 * q + j]));
                }
                const float mn = fmaxf(m, mt);
                if (ovf) {
                    if (mn == -INFINITY) {
                        ts = 0.f;
                    } else {
                        s = (m == -INFINITY) ? 0.f : s * ex2f(m - mn);
                        m = mn;
                    }
                }
                float ts2 = 0.f;
#pragma unroll 1
                for (int q = 0; q < TC_N / 32; ++q) {
                    float v[32];
                    tmem_ld32(tb + 32u * (uint32_t)q, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) ts2 += ex2f(fmaf(v[j], tk, cb[32 * q + j]) - m);
                }
                if (ovf && mn > -INFINITY) ts = ts2;
            }
            s += ts;
            if (SL) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(S.bar(BAR_ACCEMPTY(wg, u)));
                    mbar_arrive(S.bar(BAR_BEMPTY(u)));
                }
            } else {
                tc_release(S, wg, lt);
            }
        }
    }

    // ---------------- all roles done: free TMEM, combine, finalise -------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (*abort) {
        m = NAN;
        s = NAN;
        if (threadIdx.x == 0) atomicOr(p.status, SOT_DEV_TIMEOUT);
    }
    if (p.split > 1) {
        const size_t stride = (size_t)p.B * p.nr;
        if (erow) {
            p.part_m[ch * stride + rbase + row] = m;
            p.part_s[ch * stride + rbase + row] = s;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(&p.counters[b * p.rowtiles + rb], 1u);
            misc[3] = (prev == (unsigned)(p.split - 1));
        }
        __syncthreads();
        if (!misc[3]) return;
        __threadfence();
        if (erow) {
            float M = -INFINITY, Sm = 0.f;
            bool nan = false;
            for (int c = 0; c < p.split; ++c) {
                const float pm = __ldcg(p.part_m + c * stride + rbase + row);
                const float ps = __ldcg(p.part_s + c * stride + rbase + row);
                if (pm != pm || ps != ps) nan = true;
                lse_combine(M, Sm, pm, ps);
            }
            m = nan ? NAN : M;
            s = nan ? NAN : Sm;
        }
        if (threadIdx.x == 0) p.counters[b * p.rowtiles + rb] = 0u;
    }
    if (threadIdx.x == 0) misc[2] = 0;
    __syncthreads();
    if (erow) {
        if (m != m || s != s) {
            p.rstate_out[rbase + row] = NAN;
        } else if (s >= SOT_SUM_MIN && s < INFINITY && m > -INFINITY) {
            p.rstate_out[rbase + row] = m + log2f(s);
        } else {
            retry[atomicAdd(&misc[2], 1)] = row;
        }
    }
    tc_tail<TC_THREADS, SL ? 0 : TC_D>(p, S, erow, row, old, b, rb, rbase, cw, cst);
}

cudaError_t launch_tc_half(const TcPlan& plan, const HalfArgs& p, int h, int mode, cudaStream_t st) {
    if (mode != MODE_LSE || !tc_supported(p.d) || p.d != plan.d || plan.S != tc_slices(p.d))
        return cudaErrorInvalidValue;
    TcOps ops;
    ops.aimg = h ? plan.yop : plan.xop;
    ops.bimg = h ? plan.xop : plan.yop;
    ops.scale = plan.scale;
    ops.tiles_r = h ? plan.tiles_y : plan.tiles_x;
    ops.tiles_c = h ? plan.tiles_x : plan.tiles_y;
    ops.S = plan.S;
    ops.bias = plan.bias;
    ops.bias_img = nullptr;
    tc_fill_waits(ops);
    {
        const cudaError_t eb = launch_tc_bias(plan, p, ops.tiles_c, st);
        if (eb != cudaSuccess) return eb;
    }
    dim3 grid(p.rowtiles * p.split, p.B), block(TC_THREADS);
    cudaError_t e;
    if (plan.S == 1) {
        e = cudaFuncSetAttribute(tc_half_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
        if (e != cudaSuccess) return e;
        count_launches(1);
        tc_half_kernel<false><<<grid, block, TC_SMEM, st>>>(p, ops);
    } else {
        e = cudaFuncSetAttribute(tc_half_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
        if (e != cudaSuccess) return e;
        count_launches(1);
        tc_half_kernel<true><<<grid, block, TC_SMEM, st>>>(p, ops);
    }
    return cudaGetLastError();
}

// ---- the screened half-step -----------------------------------------------------------
// At the scales the half-step is used on, a row's log-sum-exp is carried by a
// handful of columns: every other term lies many binary orders below the
// row's sum.  The screened half-step scores every pair with the hi * hi
// products alone (one third of the product work of the full half-step) and
// evaluates exactly only the pairs that can matter:
//   t~_ij = tk acc_ij  with acc the fp32 accumulation of hi * hi plus the
//   column bias c_j / tk (added by a fifth MMA step, see the bias image);
//   |t~_ij - t_ij| <= Mg, from the norms of the hi parts and the residuals
//   (Cauchy-Schwarz on x.y - hx.hy = rx.hy + hx.ry + rx.ry) and fp32
//   accumulation terms, where t_ij is the exact score.
// A lower bound of the row's new value is Lb = max(L_old + lo, runmax - Mg):
// lo is the largest drop of any column bias since the row's last half-step
// (gathered by the other side), runmax the largest screened score seen so far.
// A pair is kept when t~_ij > Lb - theta - Mg; every pair dropped has
// t_ij < L_new - theta, so the dropped mass is below nc * 2^-theta of the sum,
// with theta = 26 + log2(nc): 2^-26 relative.
// Tiles are 256 columns wide (128 x 256 x 16 MMAs); each of the two row tiles
// has one 256-column accumulator, read by all sixteen epilogue warps (64
// columns of 32 rows each, with reducing loads that also give each 32-column
// chunk's maximum) and freed as soon as they hold it in registers.  Kept pairs
// go to the epilogue warp's own segment of the CTA's pool, slots numbered by
// ballot.  The CTA that finishes the row block evaluates the pools of all its
// column chunks flattened over its threads (exact scores: compensated fp32
// dot products, float-float combination), takes per-row maxima with
// shared-memory atomics and the per-row sums in 2^-48 fixed point (integer
// adds: the result does not depend on the order).  A row with a pair that did
// not fit in its segment takes the exact full-row LSE.
constexpr int SC_RETRY_INLINE = 8;  // lost rows a row block retries itself when on probation
constexpr int SC_EPI = 16;                     // epilogue warps
constexpr int SC_THREADS = 32 * (2 + SC_EPI);  // producer, MMA, epilogue
constexpr int SC_COLS = 4 * SC_N / SC_EPI;     // columns of a tile each epilogue warp screens (64)
constexpr int SC_NQ = SC_COLS / 32;            // 32-column chunks per warp and row tile
constexpr int TC_POOL = 4096;  // kept pairs per CTA
constexpr int SC_SEGS = SC_EPI;  // pool segments per CTA, one per epilogue warp
constexpr int SC_SEG = TC_POOL / SC_SEGS;
static_assert(SC_COLS % 32 == 0 && 4 * SC_N == SC_EPI * SC_COLS, "epilogue column split");
int tc_screen_pool_cap() { return TC_POOL; }
int tc_screen_pool_segments() { return SC_SEGS; }
constexpr int TC_XS = TC_D + 4;  // row stride of the fp32 row tile in shared memory (bank spread)
// Finaliser shared memory (the ring's space): the block's fp32 rows (NS = 1
// only; wider rows are read from global memory), per-row words, the segment
// offsets, then a dense copy of the kept pairs when they fit.
template <int NS>
struct ScFin {
    static constexpr uint32_t SX = NS == 1 ? TC_ROWS * TC_XS * 4 : 0;
    static constexpr uint32_t LIST = (SX + TC_ROWS * 20 + (64 * SC_SEGS + 1) * 4 + 15) & ~15u;
    static constexpr int CAP = 8192;
};
static_assert(ScFin<1>::LIST + ScFin<1>::CAP * 8 <= ScLayout<1>::NST * ScLayout<1>::STAGE &&
                  ScFin<2>::LIST + ScFin<2>::CAP * 8 <= ScLayout<2>::NST * ScLayout<2>::STAGE &&
                  ScFin<3>::LIST + ScFin<3>::CAP * 8 <= ScLayout<3>::NST * ScLayout<3>::STAGE &&
                  ScFin<4>::LIST + ScFin<4>::CAP * 8 <= ScLayout<4>::NST * ScLayout<4>::STAGE &&
                  ScFin<8>::LIST + ScFin<8>::CAP * 8 <= ScLayout<8>::NST * ScLayout<8>::STAGE &&
                  ScFin<16>::LIST + ScFin<16>::CAP * 8 <= ScLayout<16>::NST * ScLayout<16>::STAGE,
              "finaliser shared memory");

// Producer of the screened half-step: the hi halves of the CTA's two row
// tiles (every slice) once, then per 256-column tile and slice of K = 64 the
// hi halves of its two 128-point image tiles (back to back: one 256-row
// K-major operand), with the tile's bias block on its last slice.
// t0: first 128-point image tile of the chunk (even); nt: 256-column tiles.
template <int NS>
__device__ void sc_producer(const TcSmem& S, const TcOps& ops, int b, int rb, int t0, int nt) {
    using L = ScLayout<NS>;
    const int lane = threadIdx.x & 31;
    volatile int* abort = S.abort();
    int issued = 0;
    if (lane == 0) {
        if (L::STREAM) {
            mbar_arrive(S.bar(BAR_A()));  // nothing resident: the wait on the row tiles passes at once
        } else {
            mbar_arrive_expect_tx(S.bar(BAR_A()), 2 * NS * TILE_BYTES);
            for (int r = 0; r < 2; ++r)
                for (int k = 0; k < NS; ++k) {
                    const unsigned char* src = ops.aimg + (((size_t)b * ops.tiles_r + 2 * rb + r) * NS + k) * OP_BYTES;
                    bulk_g2s(S.sbase + L::OFF_A + (uint32_t)(r * NS + k) * TILE_BYTES, src, TILE_BYTES,
                             S.bar(BAR_A()));
                }
        }
    }
    const unsigned char* bimg = ops.bimg + (size_t)b * ops.tiles_c * NS * OP_BYTES;
    const unsigned char* gbias = ops.bias_img + (size_t)b * (ops.tiles_c / 2) * SC_BT;
    bool ok = true;
    for (int lt = 0; ok && lt < nt; ++lt) {
        if (lt == ops.hold_tile) break;
        for (int k = 0; k < NS; ++k) {
            const int it = lt * NS + k;
            const int st = it % L::NST;
            const uint32_t ph = (uint32_t)(it / L::NST) & 1u;
            if (!mbar_wait_bounded(S.bar(BAR_EMPTY(st)), ph ^ 1u, abort, ops.wait_ns)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = S.sbase + L::OFF_B + (uint32_t)st * L::STAGE;
                const bool last = (k == NS - 1);
                mbar_arrive_expect_tx(S.bar(BAR_FULL(st)),
                                      (L::STREAM ? 4 : 2) * TILE_BYTES + (last ? SC_BT : 0u));
                if (L::STREAM)  // slice k of both row tiles
                    for (int r = 0; r < 2; ++r)
                        bulk_g2s(dst + (uint32_t)r * TILE_BYTES,
                                 ops.aimg + (((size_t)b * ops.tiles_r + 2 * rb + r) * NS + k) * OP_BYTES, TILE_BYTES,
                                 S.bar(BAR_FULL(st)));
                bulk_g2s(dst + L::ST_B, bimg + ((size_t)(t0 + 2 * lt) * NS + k) * OP_BYTES, TILE_BYTES,
                         S.bar(BAR_FULL(st)));
                bulk_g2s(dst + L::ST_B + TILE_BYTES, bimg + ((size_t)(t0 + 2 * lt + 1) * NS + k) * OP_BYTES,
                         TILE_BYTES, S.bar(BAR_FULL(st)));
                if (last)
                    bulk_g2s(dst + L::ST_BIAS, gbias + (size_t)(t0 / 2 + lt) * SC_BT, SC_BT, S.bar(BAR_FULL(st)));
            }
            issued = it + 1;
        }
    }
    tc_producer_drain(S, issued, ops.wait_ns, L::NST);
}

// MMA warp of the screened half-step (one thread): per 256-column tile and
// row tile r, four 128 x 256 x 16 hi*hi MMAs per slice of K = 64, then the
// bias step (row-side constants times the tile's bias block), into the row
// tile's accumulator (TMEM columns 256 r ..); the epilogue frees it after
// loading it.  The thread shares its SM sub-partition with busy epilogue
// warps, so the work between two groups is kept short: descriptors are
// formed by adding offsets, and the commit that frees a stage is issued
// after the next stage's first group, off the path from one group to the next.
template <int NS>
__device__ void sc_mma(const TcSmem& S, uint32_t tmem, int nt, uint64_t wait_ns) {
    using L = ScLayout<NS>;
    if ((threadIdx.x & 31) == 0) {
        volatile int* abort = S.abort();
        bool ok = mbar_wait_bounded(S.bar(BAR_A()), 0u, abort, wait_ns);
        bool issued_any = false;
        const uint32_t idesc = f16_idesc(TC_M, SC_N);
        // Descriptors: the start address field (bits 0-13, address / 16) is the
        // only part that differs, and every address here is below 256 KB, so a
        // byte offset o is added to a descriptor as o / 16 with no carry out of
        // the field; it advances by 2 per K = 16 step (32 bytes).
        const uint64_t adesc0 = sw128_desc(S.sbase + (L::STREAM ? L::OFF_B : L::OFF_A)),
                       acdesc0 = sw32_desc(S.sbase + L::OFF_AC);
        const uint64_t bdesc0 = sw128_desc(S.sbase + L::OFF_B + L::ST_B),
                       bbdesc0 = sw32_desc(S.sbase + L::OFF_B + L::ST_BIAS);
        int prev_st = -1;
        for (int lt = 0; ok && lt < nt; ++lt) {
            for (int k = 0; ok && k < NS; ++k) {
                const int it = lt * NS + k;
                const int st = it % L::NST;
                const uint32_t ph = (uint32_t)(it / L::NST) & 1u;
                if (!mbar_wait_bounded(S.bar(BAR_FULL(st)), ph, abort, wait_ns)) {
                    ok = false;
                    break;
                }
                for (int r = 0; r < 2; ++r) {
                    if (k == 0) {
                        if (!mbar_wait_bounded(S.bar(BAR_ACCEMPTY(r, 0)), ((uint32_t)lt & 1u) ^ 1u, abort, wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    issued_any = true;
                    const uint32_t d = tmem + (uint32_t)(r * SC_N);
                    const uint64_t ad = adesc0 + (uint64_t)(L::STREAM ? st * (L::STAGE >> 4) + r * (TILE_BYTES >> 4)
                                                                      : (r * NS + k) * (TILE_BYTES >> 4));
                    const uint64_t bd = bdesc0 + (uint64_t)(st * (L::STAGE >> 4));
#pragma unroll
                    for (int kk = 0; kk < TC_D / 16; ++kk)
                        tc_mma_f16(d, ad + 2u * (uint64_t)kk, bd + 2u * (uint64_t)kk, idesc, (k > 0 || kk > 0) ? 1u : 0u);
                    if (k == NS - 1) {
                        tc_mma_f16(d, acdesc0 + (uint64_t)(r * (SC_AT >> 4)),
                                   bbdesc0 + (uint64_t)(st * (L::STAGE >> 4)), idesc, 1u);
                        tc_commit(S.bar(BAR_ACCFULL(r, 0)));
                    }
                    if (r == 0 && prev_st >= 0) {
                        // the previous stage: its last readers were issued before this group
                        tc_commit(S.bar(BAR_EMPTY(prev_st)));
                        prev_st = -1;
                    }
                }
                if (!ok) break;
                prev_st = st;
            }
        }
        if (prev_st >= 0) tc_commit(S.bar(BAR_EMPTY(prev_st)));
        tc_mma_drain(S, issued_any, wait_ns);
    }
    __syncwarp();
}

struct TcScreenK {
    uint2* pool;
    int pool_cap;
    int* pool_cnt;
    int* lost;
    int* ovf;
    const unsigned* nrm_r;  // [B][4] with the row side's (hi, residual) pair first
    const unsigned* nrm_c;  // column side's pair at the same stride
    const unsigned* cmax;   // [B] max |c_j| of this half-step's column biases (float bits)
};

// Per-chunk maxima of one row over NQ x 32 columns of a tile, from the
// accumulators (raw bits; accumulator units, biases included): one
// three-input max chain per 32-column chunk.
// Screen NQ x 32 columns of one row (accumulator bits in r, columns jt ..):
// the per-chunk maxima raise the running maximum, and every pair of a chunk
// that reaches the threshold goes to the CTA's pool.
struct ScShared {  // the same for every row of the warp
    float Mg, tk, inv_tk;
    uint2* seg;   // this warp's pool segment
    int wcount;   // entries reserved in it (warp-uniform)
    const float* ycol;  // the columns' fp32 coordinates (the finaliser reads a kept pair's row)
    int nc, d;
};
struct ScRow {  // one row's screening state
    float Lb, off, runmax;
    int* lost;   // this row's "lost" word
    unsigned rl; // row within the row block
    bool erow;
};
// mq[q]: the maximum of chunk q, formed by the TMEM load itself.
template <int NQ>
__device__ __forceinline__ void sc_screen(const uint32_t (&r)[NQ][32], const uint32_t (&mqb)[NQ], int jt,
                                          ScShared& c, ScRow& s) {
    float mq[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) mq[q] = __uint_as_float(mqb[q]);
    // thresholds in accumulator units (score = tk * acc, tk > 0)
    float mall = mq[0];
#pragma unroll
    for (int q = 1; q < NQ; ++q) mall = fmaxf(mall, mq[q]);
    s.runmax = fmaxf(s.runmax, c.tk * mall);
    // (a reciprocal, not a division: the margin absorbs its rounding)
    const float Ta = (fmaxf(s.Lb, s.runmax - c.Mg) - s.off) * c.inv_tk;
    bool hq[NQ];
    bool hit = false;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        hq[q] = s.erow && mq[q] > Ta;
        hit = hit || hq[q];
    }
    if (!__any_sync(0xffffffffu, hit)) return;
    const unsigned lt_mask = (1u << (threadIdx.x & 31)) - 1u;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        if (!__any_sync(0xffffffffu, hq[q])) continue;
        unsigned pm = 0u;  // this lane's kept columns of the chunk
        if (hq[q]) {
            // bit j = sign of Ta - v_j: set exactly when v_j > Ta (a -inf or NaN
            // score gives +inf or a positive NaN: never set); four independent
            // 8-bit chains
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                unsigned mg = 0u;
#pragma unroll
                for (int j = 7; j >= 0; --j)
                    mg = __funnelshift_l(__float_as_uint(__fsub_rn(Ta, __uint_as_float(r[q][8 * g + j]))), mg, 1);
                pm |= mg << (8 * g);
            }
        }
        // Slots of the warp's segment, one pair per lane and round, numbered by
        // lane order (ballot + popc): dense, so every slot below the capacity that
        // is counted is written.  A pair past the capacity loses its row.
        for (;;) {
            const unsigned act = __ballot_sync(0xffffffffu, pm != 0u);
            if (act == 0u) break;
            if (pm) {
                const int j = __ffs(pm) - 1;
                pm &= pm - 1u;
                const int slot = c.wcount + __popc(act & lt_mask);
                const int jc = jt + 32 * q + j;
                if (slot < SC_SEG) {
                    c.seg[slot] = make_uint2((unsigned)jc, s.rl);
                    if (jc < c.nc) {  // the finaliser reads this column's row: bring it into L2 now
                        const float* yr = c.ycol + (size_t)jc * c.d;
                        for (int o = 0; o < c.d; o += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(yr + o));
                    }
                } else {
                    *s.lost = 1;
                }
            }
            c.wcount += __popc(act);
        }
    }
}

// 18 warps put five on one SM sub-partition, whose 16384 registers then allow
// 96 per thread.
template <int NS>
__global__ void __launch_bounds__(SC_THREADS, 1) tc_screen_kernel(HalfArgs p, TcOps ops, TcScreenK sk) {
    using L = ScLayout<NS>;
    using F = ScFin<NS>;
    constexpr int D = NS * TC_D;  // coordinates (the images' K)
    if (p.stop_flag && *(volatile const int*)p.stop_flag) return;
    extern __shared__ unsigned char smem_raw[];
    const TcSmem S = tc_smem(smem_raw, L::OFF_HDR);
    int* misc = S.misc();
    volatile int* abort = S.abort();
    int* retry = S.retry();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int rb = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rb * TC_ROWS;
    const int c_begin = ch * p.chunk;  // a multiple of SC_N
    const int c_end = min(p.nc, c_begin + p.chunk);
    const int t0 = c_begin / TC_N;
    const int nt = (c_end - c_begin + SC_N - 1) / SC_N;  // 256-column tiles
    const float* cw = p.cw2 + (size_t)b * p.nc;
    const float* cst = p.cstate + (size_t)b * p.nc;
    const size_t rbase = (size_t)b * p.nr;
    const float sc = ops.scale[b];
    const float tk = p.two_kappa / (sc * sc);
    const size_t cta0 = ((size_t)b * p.rowtiles + rb) * p.split;  // first pool of this row block

    if (p.lo_reset && blockIdx.x == 0 && blockIdx.y == 0)
        for (int k = threadIdx.x; k < p.B; k += SC_THREADS) p.lo_reset[k] = SOT_ORD_EMPTY;
    // Row-side constants of the bias step, (2^E, 2^(E-11), 2^(E-22), 0, ...) in
    // K = 0..15 of every row of both row tiles.  A cloud whose biases need
    // E > 15 is not screened: its rows take the exact LSE.
    const int E = tc_bias_exp(sk.cmax[b], sc, p.two_kappa);
    const bool screenable = E <= 15;
    const int nts = screenable ? nt : 0;  // tiles this CTA screens
    if (screenable) {
        const unsigned h0 = __half_as_ushort(__float2half_rn(ldexpf(1.f, E)));
        const unsigned h1 = __half_as_ushort(__float2half_rn(ldexpf(1.f, E - 11)));
        const unsigned h2 = __half_as_ushort(__float2half_rn(ldexpf(1.f, E - 22)));
        const uint4 c0 = make_uint4(h0 | (h1 << 16), h2, 0u, 0u), z = make_uint4(0u, 0u, 0u, 0u);
        for (int e = threadIdx.x; e < 2 * TC_M * 2; e += SC_THREADS) {
            const int rt = e / (2 * TC_M), r = (e % (2 * TC_M)) >> 1, c = e & 1;
            *reinterpret_cast<uint4*>(S.sm + L::OFF_AC + rt * SC_AT + sw32_offset(r, 8 * c)) = c ? z : c0;
        }
        fence_proxy_async_smem();
    }
    // stages are freed by the MMA commit alone; every accumulator is read by all 16 epilogue warps
    const uint32_t tmem = tc_setup(S, warp, 1, SC_EPI);

    const int q4 = warp & 3;  // the TMEM lane quarter this warp may access
    // the row this thread finalises (and whose marginal-error term it forms):
    // warps 2..9, row tile (warp - 2) / 4
    const int row = row0 + ((warp - 2) >> 2) * TC_M + q4 * 32 + lane;
    const bool erow = (warp >= 2) && (warp < 10) && row < p.nr;
    const float old = (erow && p.rstate_in) ? p.rstate_in[rbase + row] : 0.f;

    if (warp == 0) {
        sc_producer<NS>(S, ops, b, rb, t0, nts);
    } else if (warp == 1) {
        sc_mma<NS>(S, tmem, nts, ops.wait_ns);
    } else {
        // Screening: epilogue warp ew = warp - 2 (column group cg = ew / 4, lane
        // quarter q4) reads columns SC_COLS cg .. of both row tiles' accumulators for
        // TMEM lanes 32 q4 ..: rows row0 + 32 q4 + lane (tile 0) and row0 + 128 +
        // 32 q4 + lane (tile 1).  An accumulator is freed as soon as all SC_EPI warps
        // have loaded their share, before the screening arithmetic.
        const int ew = warp - 2, cg = ew >> 2;
        if (!screenable && erow) sk.lost[rbase + row] = 1;
        // screening margin of this cloud (scaled units -> log2 units); the
        // last term covers the fp32 rounding of the biases held in the
        // accumulator and of the products added onto them
        const float hr = __uint_as_float(sk.nrm_r[4 * b]), rr = __uint_as_float(sk.nrm_r[4 * b + 1]);
        const float hc = __uint_as_float(sk.nrm_c[4 * b]), rc = __uint_as_float(sk.nrm_c[4 * b + 1]);
        const float cmax = __uint_as_float(sk.cmax[b]);
        ScShared c;
        c.Mg = 1.01f * tk * (rr * hc + hr * rc + rr * rc + (float)NS * 1.5258789e-5f * hr * hc) + 1.5258789e-5f * cmax +
               0.02f;
        c.tk = tk;
        c.inv_tk = 1.f / tk;
        c.seg = sk.pool + ((cta0 + ch) * SC_SEGS + ew) * (size_t)SC_SEG;
        c.wcount = 0;
        c.ycol = p.cpack + (size_t)b * p.nc * D;
        c.nc = p.nc;
        c.d = D;
        const float theta_off = 26.f + log2f((float)p.nc) + c.Mg + 0.05f;
        const float lo = (!p.cold && p.lo_in) ? ord_decode(p.lo_in[b]) : -INFINITY;
        ScRow s[2];
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
            const int rrow = row0 + rt * TC_M + q4 * 32 + lane;
            const bool ok_row = rrow < p.nr;
            const float o = (ok_row && p.rstate_in) ? p.rstate_in[rbase + rrow] : 0.f;
            s[rt].off = theta_off + 1.5e-5f * fabsf(o);
            s[rt].Lb = isfinite(lo) ? o + lo : -INFINITY;
            s[rt].runmax = -INFINITY;
            s[rt].lost = sk.lost + rbase + (ok_row ? rrow : 0);
            s[rt].rl = (unsigned)(rt * TC_M + q4 * 32 + lane);
            s[rt].erow = ok_row;
        }
        const uint32_t tq = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(cg * SC_COLS);  // lanes, columns
        bool ok = true;
        for (int lt = 0; ok && lt < nts; ++lt) {
#pragma unroll
            for (int rt = 0; rt < 2; ++rt) {
                if (!mbar_wait_bounded(S.bar(BAR_ACCFULL(rt, 0)), (uint32_t)lt & 1u, abort, ops.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the loads reduce each lane's 32 columns to their maximum on the way
                uint32_t r[SC_NQ][32], mq[SC_NQ];
#pragma unroll
                for (int q = 0; q < SC_NQ; ++q)
                    tmem_ld32_max_issue(tq + (uint32_t)(rt * SC_N) + 32u * (uint32_t)q, r[q], mq[q]);
#pragma unroll
                for (int q = 0; q < SC_NQ; ++q) tmem_wait_ld_max(r[q], mq[q]);
                // this warp's share of the accumulator is in registers: free it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(S.bar(BAR_ACCEMPTY(rt, 0)));
                sc_screen<SC_NQ>(r, mq, c_begin + lt * SC_N + SC_COLS * cg, c, s[rt]);
            }
        }
        if (lane == 0) sk.pool_cnt[(cta0 + ch) * SC_SEGS + ew] = min(c.wcount, SC_SEG);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (*abort) {
        if (erow) sk.lost[rbase + row] = 2;  // poisoned
        if (threadIdx.x == 0) atomicOr(p.status, SOT_DEV_TIMEOUT);
    }
    // (pool_cnt: written by each epilogue warp for its segment)
    if (p.split > 1) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(&p.counters[b * p.rowtiles + rb], 1u);
            misc[3] = (prev == (unsigned)(p.split - 1));
        }
        __syncthreads();
        if (!misc[3]) return;
        __threadfence();
        if (threadIdx.x == 0) p.counters[b * p.rowtiles + rb] = 0u;
    }

    // ---------------- finish the row block: exact scores of the kept pairs ----------------
    float* sx = reinterpret_cast<float*>(S.sm + L::OFF_B);                  // [TC_ROWS][TC_XS] fp32 rows (NS = 1)
    float* s_ref = reinterpret_cast<float*>(S.sm + L::OFF_B + F::SX);       // [TC_ROWS] reference L_old
    unsigned* s_max = reinterpret_cast<unsigned*>(s_ref + TC_ROWS);          // [TC_ROWS] ord-encoded max
    unsigned long long* s_sum = reinterpret_cast<unsigned long long*>(s_max + TC_ROWS);  // [TC_ROWS] fixed point
    int* s_lost = reinterpret_cast<int*>(s_sum + TC_ROWS);                   // [TC_ROWS]
    int* s_off = s_lost + TC_ROWS;                                           // [split * SC_SEGS + 1]
    {
        if (NS == 1) {
            // the block's fp32 rows: every load issued before the first store
            const float4* src = reinterpret_cast<const float4*>(p.rpack + rbase * TC_D);
            constexpr int NE = TC_ROWS * (TC_D / 4), NL = (NE + SC_THREADS - 1) / SC_THREADS;
            float4 buf[NL];
#pragma unroll
            for (int i = 0; i < NL; ++i) {
                const int e = threadIdx.x + i * SC_THREADS, rg = row0 + e / (TC_D / 4);
                buf[i] = (e < NE && rg < p.nr) ? __ldg(src + (size_t)rg * (TC_D / 4) + e % (TC_D / 4))
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < NL; ++i) {
                const int e = threadIdx.x + i * SC_THREADS;
                if (e < NE) *reinterpret_cast<float4*>(sx + (e / (TC_D / 4)) * TC_XS + 4 * (e % (TC_D / 4))) = buf[i];
            }
        }
        for (int r = threadIdx.x; r < TC_ROWS; r += SC_THREADS) {
            const int rg = row0 + r;
            float ref = 0.f;
            int lost = 0;
            if (rg < p.nr) {
                const float o = p.rstate_in ? p.rstate_in[rbase + rg] : 0.f;
                ref = isfinite(o) ? o : 0.f;
                lost = __ldcg(sk.lost + rbase + rg);
                if (lost) {
                    sk.lost[rbase + rg] = 0;
                    atomicAdd(&misc[5], 1);
                }
            }
            s_ref[r] = ref;
            s_max[r] = 0u;  // below the encoding of every float
            s_sum[r] = 0ull;
            s_lost[r] = lost;
        }
        // the block's pool segments (every chunk's): sizes ...
        for (int g = threadIdx.x; g < p.split * SC_SEGS; g += SC_THREADS)
            s_off[g + 1] = __ldcg(sk.pool_cnt + cta0 * SC_SEGS + g);
    }
    __syncthreads();
    // On probation (p.redo set): a row block with more lost rows than the
    // one-row retry handles writes nothing and is left to the full half-step
    // launched next (its rows keep their old values, which that step reads).
    if (p.redo && misc[5] > SC_RETRY_INLINE) {
        if (threadIdx.x == 0) {
            p.redo[(size_t)b * p.rowtiles + rb] = 1;
            atomicAdd(sk.ovf, misc[5]);
        }
        return;
    }
    const int nseg = p.split * SC_SEGS;
    if (warp == 0) {  // ... and their prefix sums (segment g holds entries s_off[g] .. s_off[g + 1])
        int carry = 0;
        for (int g0 = 0; g0 < nseg; g0 += 32) {
            int v = (g0 + lane < nseg) ? s_off[g0 + lane + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (g0 + lane < nseg) s_off[g0 + lane + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_off[0] = 0;
    }
    __syncthreads();
    const int total = s_off[nseg];
    const float4* ybase = reinterpret_cast<const float4*>(p.cpack + (size_t)b * p.nc * D);
    // the kept pairs, segment after segment, into one dense list in shared
    // memory when they fit (every later lookup is one shared load)
    uint2* s_list = reinterpret_cast<uint2*>(S.sm + L::OFF_B + F::LIST);
    const bool dense = total <= F::CAP;
    if (dense) {
        for (int g = warp; g < nseg; g += SC_THREADS / 32) {
            const uint2* src = sk.pool + (cta0 * SC_SEGS + g) * (size_t)SC_SEG;
            const int o = s_off[g], cnt = s_off[g + 1] - o;
            for (int i = lane; i < cnt; i += 32) s_list[o + i] = __ldcg(src + i);
        }
        __syncthreads();
    }
    // pass 1: exact score of every kept pair, relative to the row's reference;
    // row maxima.
    auto entry = [&](int k) -> uint2* {  // the dense list, or segment g with s_off[g] <= k < s_off[g + 1]
        if (dense) return s_list + k;
        int lo = 0, hi = nseg;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= k) lo = mid; else hi = mid;
        }
        return sk.pool + (cta0 * SC_SEGS + lo) * (size_t)SC_SEG + (k - s_off[lo]);
    };
    // Four lanes per kept pair (a quad), each taking a quarter of every slice of 64:
    // short dependency chains and few live registers.  The quad's partial
    // dot products are error-free float-float values (Dekker / Knuth
    // transformations, errors summed alongside), combined across the quad
    // by shuffles; lane 0 of the quad forms
    //   t - ref = 2 kappa (sum hs + sum es) + (cw_j - cst_j) - ref
    // in float-float arithmetic (the fp64 pipe is slow here): the large parts
    // cancel exactly, the small ones are added last.
    constexpr int QD = TC_D / 4;  // coordinates per lane of a quad
    const int sub = lane & 3;
    for (int k0 = 0; k0 < total; k0 += SC_THREADS / 4) {
        const int k = k0 + (threadIdx.x >> 2);
        const bool in = k < total;
        uint2* e0 = in ? entry(k) : nullptr;
        const uint2 it0 = in ? (dense ? *e0 : __ldcg(e0)) : make_uint2(0u, 0u);
        const bool v0 = in && !s_lost[it0.y] && (int)it0.x < p.nc;
        float hs[4] = {0.f, 0.f, 0.f, 0.f}, es[4] = {0.f, 0.f, 0.f, 0.f};
        if (v0) {
            // x: the staged row (NS = 1) or the row in global memory
            const float* xrow = (NS == 1) ? sx + it0.y * TC_XS : p.rpack + (rbase + row0 + it0.y) * (size_t)D;
#pragma unroll 1
            for (int sl = 0; sl < NS; ++sl) {
                const float4* y = ybase + (size_t)it0.x * (D / 4) + sl * (TC_D / 4) + sub * (QD / 4);
                const float* xr = xrow + sl * TC_D + sub * QD;
                float4 yv[QD / 4];
#pragma unroll
                for (int q = 0; q < QD / 4; ++q) yv[q] = __ldg(y + q);
#pragma unroll
                for (int q = 0; q < QD / 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(xr + 4 * q);
                    const float xa[4] = {x.x, x.y, x.z, x.w};
                    const float ya[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float2 pr = two_prod(xa[w], ya[w]);
                        const float2 sn = two_sum(hs[w], pr.x);
                        hs[w] = sn.x;
                        es[w] = __fadd_rn(es[w], __fadd_rn(pr.y, sn.y));
                    }
                }
            }
        }
        // this lane's partial as one float-float value (S, E) ...
        const float2 s01 = two_sum(hs[0], hs[1]), s23 = two_sum(hs[2], hs[3]);
        float2 S2 = two_sum(s01.x, s23.x);
        float E2 = __fadd_rn(__fadd_rn(__fadd_rn(es[0], es[1]), __fadd_rn(es[2], es[3])),
                             __fadd_rn(__fadd_rn(s01.y, s23.y), S2.y));
        float Sv = S2.x;
        // ... then the quad's (every lane of the warp takes part in the shuffles)
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            const float So = __shfl_xor_sync(0xffffffffu, Sv, o);
            const float Eo = __shfl_xor_sync(0xffffffffu, E2, o);
            const float2 t = two_sum(Sv, So);
            Sv = t.x;
            E2 = __fadd_rn(__fadd_rn(E2, Eo), t.y);
        }
        if (in && sub == 0) {
            if (v0) {
                const int rl = (int)it0.y, j = (int)it0.x;
                const float2 P2 = two_prod(p.two_kappa, Sv);
                const float2 C2 = two_sum(cw[j], -cst[j]);
                const float2 U2 = two_sum(P2.x, C2.x);
                const float2 V2 = two_sum(U2.x, -s_ref[rl]);
                const float trel = __fadd_rn(
                    V2.x, __fadd_rn(__fadd_rn(V2.y, U2.y), __fadd_rn(__fadd_rn(P2.y, C2.y), __fmul_rn(p.two_kappa, E2))));
                e0->x = __float_as_uint(trel);
                atomicMax(s_max + rl, ord_encode(trel));
            } else if (!s_lost[it0.y]) {
                e0->x = __float_as_uint(-INFINITY);
            }
        }
    }
    __syncthreads();
    // pass 2: row sums in 2^-48 fixed point (each term <= 1), four entries per round
    for (int k0 = threadIdx.x; k0 < total; k0 += 4 * SC_THREADS) {
        uint2 it[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * SC_THREADS;
            it[u] = (k < total) ? (dense ? s_list[k] : __ldcg(entry(k))) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u * SC_THREADS;
            const int rl = (int)it[u].y;
            if (k >= total || s_lost[rl]) continue;
            const float w = ex2f(__uint_as_float(it[u].x) - ord_decode(s_max[rl]));
            atomicAdd(s_sum + rl, (unsigned long long)__float2ull_rn(w * 281474976710656.f));
        }
    }
    if (threadIdx.x == 0) misc[2] = 0;
    __syncthreads();
    if (erow) {
        const int rl = row - row0;
        if (s_lost[rl] == 2) {
            p.rstate_out[rbase + row] = NAN;
        } else if (s_lost[rl]) {
            retry[atomicAdd(&misc[2], 1)] = row;
            atomicAdd(sk.ovf, 1);
        } else if (s_sum[rl] == 0ull) {
            p.rstate_out[rbase + row] = -INFINITY;
        } else {
            p.rstate_out[rbase + row] =
                s_ref[rl] + (ord_decode(s_max[rl]) + (log2f(__ull2float_rn(s_sum[rl])) - 48.f));
        }
    }
    tc_tail<SC_THREADS, NS == 1 ? TC_D : 0>(p, S, erow, row, old, b, rb, rbase, cw, cst);
}

cudaError_t launch_tc_screen(const TcPlan& plan, const HalfArgs& p, int h, const TcScreen& sc, cudaStream_t st) {
    if (!tc_supported(p.d) || p.d != plan.d || !p.lo_in || !sc.pool || !sc.pool_cnt || !sc.lost ||
        sc.pool_cap != TC_POOL)
        return cudaErrorInvalidValue;
    TcOps ops;
    ops.aimg = h ? plan.yop : plan.xop;
    ops.bimg = h ? plan.xop : plan.yop;
    ops.scale = plan.scale;
    ops.tiles_r = h ? plan.tiles_y : plan.tiles_x;
    ops.tiles_c = h ? plan.tiles_x : plan.tiles_y;
    ops.S = plan.S;
    ops.bias = plan.bias;
    ops.bias_img = plan.bimg;
    tc_fill_waits(ops);
    {
        const cudaError_t eb = launch_tc_bias_image(plan, p, ops.tiles_c, st);
        if (eb != cudaSuccess) return eb;
    }
    TcScreenK sk;
    sk.cmax = plan.cmax + 2 * p.B;
    sk.pool = sc.pool;
    sk.pool_cap = sc.pool_cap;
    sk.pool_cnt = sc.pool_cnt;
    sk.lost = sc.lost;
    sk.ovf = sc.ovf;
    sk.nrm_r = plan.nrm + (h ? 2 : 0);
    sk.nrm_c = plan.nrm + (h ? 0 : 2);
    if (p.chunk % SC_N != 0 || ops.tiles_c % 2 != 0) return cudaErrorInvalidValue;
    dim3 grid(p.rowtiles * p.split, p.B), block(SC_THREADS);
#define SOT_SC_CASE(NSV)                                                                                   \
    case NSV: {                                                                                            \
        cudaError_t e = cudaFuncSetAttribute(tc_screen_kernel<NSV>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             (int)ScLayout<NSV>::SMEM);                                    \
        if (e != cudaSuccess) return e;                                                                    \
        count_launches(1);                                                                                 \
        tc_screen_kernel<NSV><<<grid, block, ScLayout<NSV>::SMEM, st>>>(p, ops, sk);                       \
        break;                                                                                             \
    }
    switch (plan.S) {
        SOT_SC_CASE(1)
        SOT_SC_CASE(2)
        SOT_SC_CASE(3)
        SOT_SC_CASE(4)
        SOT_SC_CASE(8)
        SOT_SC_CASE(16)
        default: return cudaErrorInvalidValue;
    }
#undef SOT_SC_CASE
    return cudaGetLastError();
}

// ---- plan application (cost, gradient, row sums) ------------------------------------
// Per row i, with the final potentials and P_ij / a_i = 2^(score_ij - L_i):
//   r_i = sum_j P_ij,  q_i = sum_j P_ij C_ij,  v_i = sum_j P_ij y_j.
// r_i sums every pair.  q_i and v_i sum the pairs whose term is within 2^-40 of
// the row's running scale: an omitted term is below 2^-40 of the row mass, so
// at most m * 2^-40 of it is dropped in all.  Such pairs are a handful per row.
// Their terms are evaluated exactly (fp64, direct form, from the caller's
// coordinates and potentials): log2(P_ij / a_i) = log2 b_j + kappa (f_i + g_j - C_ij).
// In fp32 the expanded-form score rounds at the magnitude 2 kappa |x||y|
// (~1800 log2 units at d = 64, eps = 0.1), which alone moves the gradient by
// ~1e-4 relative; the exact evaluation of the significant pairs removes that.
// Pass A of a tile forms the fp32 exponentials and the row sum, and marks the
// 4-column groups that hold a significant pair; pass B revisits only those,
// replaces their fp32 terms in r_i and forms q_i and v_i.
struct TcApplyExtra {
    const float* nx;      // [B][n]
    const float* ny;      // [B][m]
    const float* X;       // [B][n][d] caller coordinates
    const float* Y;       // [B][m][d] caller coordinates
    const float* f;       // [B][n] caller potentials
    const float* g;       // [B][m]
    double kappa64;
    const float* a;       // [B][n] or NULL (uniform)
    const float* shift;   // [B][d]
    float* vpart;         // [split][B*n][d], zero on entry
    float* part_r;        // [split][B*n]
    float* part_q;        // [split][B*n]
    float* cost_part;     // [B][rowtiles] or NULL
    float* grad;          // [B][n][d] or NULL
    float* rowsum;        // [B][n] or NULL
};

constexpr float TC_SIG = -40.f;  // a pair is significant when log2(P_ij / a_i) > TC_SIG

// SL: d > 64, the operands stream in slices as in the sliced full half-step;
// a lane of pass B then owns 2 coordinates of every slice of 64.
template <bool SL>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_apply_kernel(HalfArgs p, TcOps ops, TcApplyExtra x) {
    extern __shared__ unsigned char smem_raw[];
    const TcSmem S = tc_smem(smem_raw);
    int* misc = S.misc();
    volatile int* abort = S.abort();
    float* red = S.red();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int rb = blockIdx.x / p.split, ch = blockIdx.x % p.split;
    const int row0 = rb * TC_ROWS;
    const int c_begin = ch * p.chunk;
    const int c_end = min(p.nc, c_begin + p.chunk);
    const int t0 = c_begin / TC_N;
    const int nt = (c_end - c_begin + TC_N - 1) / TC_N;
    const float* cw = p.cw2 + (size_t)b * p.nc;
    const size_t rbase = (size_t)b * p.nr;
    const float sc = ops.scale[b];
    const float tk = p.two_kappa / (sc * sc);
    const int D = SL ? p.d : TC_D;  // coordinates (a multiple of 64)
    const int ns = D / TC_D;

    const uint32_t tmem = SL ? tc_setup(S, warp, 1, 4, 8) : tc_setup(S, warp);

    float m = 0.f, r = 0.f, q = 0.f;
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int row = row0 + wg * TC_M + q4 * 32 + lane;
    const bool erow = (warp >= 2) && row < p.nr;
    float* vrow = erow ? x.vpart + (((size_t)ch * p.B * p.nr) + rbase + row) * D : nullptr;

    if (warp == 0) {
        if (SL) tc_producer_sl(S, ops, b, rb, t0, nt, ns);
        else tc_producer(S, ops, b, rb, t0, nt);
    } else if (warp == 1) {
        if (SL) tc_mma_sl(S, tmem, nt, ns, ops.wait_ns);
        else tc_mma(S, tmem, nt, ops.wait_ns);
    } else {
        const float lrow = erow ? p.rstate_in[rbase + row] : 0.f;
        m = erow ? lrow - SOT_STAB_BIAS : INFINITY;
        const float fi = erow ? x.f[rbase + row] : 0.f;
        const float2 kap = make_float2((float)x.kappa64, (float)(x.kappa64 - (double)(float)x.kappa64));
        const float* yorig = x.Y + (size_t)b * p.nc * D;
        const float* gpot = x.g + (size_t)b * p.nc;
        const float2 tk2 = make_float2(tk, tk);
        for (int lt = 0; lt < nt; ++lt) {
            const int st = lt % TC_S;
            const uint32_t ph = (uint32_t)(lt / TC_S) & 1u;
            const int u = lt & 1;
            const uint32_t pu = (uint32_t)(lt >> 1) & 1u;
            // the tile's biases: in its stage, or (sliced) in bias slot u
            if (!mbar_wait_bounded(S.bar(SL ? BAR_BFULL(u) : BAR_FULL(st)), SL ? pu : ph, abort, ops.wait_ns)) break;
            if (!mbar_wait_bounded(S.bar(BAR_ACCFULL(wg, u)), pu, abort, ops.wait_ns)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)((2 * wg + u) * TC_N);
            const float* cb = S.bias() + (SL ? u : st) * TC_N;
            // pass A: row sum, significance marks per 4-column group.  A pair is
            // significant when t - L_i > TC_SIG, i.e. e = t - m > TC_SIG + (L_i - m).
            const float2 nm2 = make_float2(-m, -m);
            const float sig_e = TC_SIG + (lrow - m);
            float2 acc2 = make_float2(0.f, 0.f);
            uint32_t sig = 0u;
#pragma unroll 1
            for (int qq = 0; qq < TC_N / 32; ++qq) {
                float v[32];
                tmem_ld32(tb + 32u * (uint32_t)qq, v);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 c4 = *reinterpret_cast<const float4*>(cb + 32 * qq + j);
                    const float2 e0 = fadd2(ffma2(make_float2(v[j], v[j + 1]), tk2, make_float2(c4.x, c4.y)), nm2);
                    const float2 e1 =
                        fadd2(ffma2(make_float2(v[j + 2], v[j + 3]), tk2, make_float2(c4.z, c4.w)), nm2);
                    acc2 = fadd2(acc2, make_float2(ex2f(e0.x), ex2f(e0.y)));
                    acc2 = fadd2(acc2, make_float2(ex2f(e1.x), ex2f(e1.y)));
                    const float emax = fmaxf(fmaxf(e0.x, e0.y), fmaxf(e1.x, e1.y));
                    sig |= (emax > sig_e) ? (1u << (8 * qq + j / 4)) : 0u;
                }
            }
            float ts = acc2.x + acc2.y;
            const bool ovf = !(ts < SOT_TILE_SUM_MAX);
            if (__any_sync(0xffffffffu, ovf)) {
                float mt = -INFINITY;
#pragma unroll 1
                for (int qq = 0; qq < TC_N / 32; ++qq) {
                    float v[32];
                    tmem_ld32(tb + 32u * (uint32_t)qq, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) mt = fmaxf(mt, fmaf(v[j], tk, cb[32 * qq + j]));
                }
                const float mn = fmaxf(m, mt);
                if (ovf && mn > m) {
                    const float f = ex2f(m - mn);
                    r *= f;
                    q *= f;
                    for (int k = 0; k < D; ++k) vrow[k] *= f;
                    m = mn;
                }
                float ts2 = 0.f;
#pragma unroll 1
                for (int qq = 0; qq < TC_N / 32; ++qq) {
                    float v[32];
                    tmem_ld32(tb + 32u * (uint32_t)qq, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) ts2 += ex2f(fmaf(v[j], tk, cb[32 * qq + j]) - m);
                }
                if (ovf) ts = ts2;
            }
            r += ts;
            // pass B: cost and barycentre terms of the significant pairs.  The warp
            // takes them one at a time: every lane owns 2 of the 64 coordinates,
            // C_ij is reduced across the warp in float-float arithmetic (the fp64
            // pipe is slow here), and the row's v_i update is one coalesced
            // 256-byte write.
            const float sig_b = TC_SIG + (lrow - m);
#pragma unroll 1
            for (int qq = 0; qq < TC_N / 32; ++qq) {
                if (!__any_sync(0xffffffffu, ((sig >> (8 * qq)) & 0xFFu) != 0u)) continue;
                float v[32];
                tmem_ld32(tb + 32u * (uint32_t)qq, v);
#pragma unroll 1
                for (int c = 0; c < 32; ++c) {
                    const int cl = 32 * qq + c;
                    const float e = fmaf(v[c], tk, cb[cl]) - m;
                    unsigned todo = __ballot_sync(0xffffffffu, erow && e > sig_b);
                    if (!todo) continue;
                    const int j = (t0 + lt) * TC_N + cl;
                    const float* yj = yorig + (size_t)j * D + 2 * lane;
                    const float gj = gpot[j], lbj = cw[j];
                    while (todo) {
                        const int l = __ffs(todo) - 1;
                        todo &= todo - 1u;
                        const int rl = __shfl_sync(0xffffffffu, row, l);
                        const float* xl = x.X + (rbase + rl) * D + 2 * lane;
                        // C_lj: exact coordinate differences, their squares to ~2^-48
                        float2 C2 = make_float2(0.f, 0.f);
                        for (int sl = 0; sl < ns; ++sl) {
                            const float2 xv = *reinterpret_cast<const float2*>(xl + sl * TC_D);
                            const float2 yv = *reinterpret_cast<const float2*>(yj + sl * TC_D);
                            const float2 d0 = two_sum(xv.x, -yv.x), d1 = two_sum(xv.y, -yv.y);
                            float2 s0 = two_prod(d0.x, d0.x), s1 = two_prod(d1.x, d1.x);
                            s0.y = __fmaf_rn(2.f * d0.x, d0.y, s0.y);
                            s1.y = __fmaf_rn(2.f * d1.x, d1.y, s1.y);
                            C2 = ff_add(C2, ff_add(s0, s1));
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1)
                            C2 = ff_add(C2, make_float2(__shfl_xor_sync(0xffffffffu, C2.x, o),
                                                        __shfl_xor_sync(0xffffffffu, C2.y, o)));
                        const float fl = __shfl_sync(0xffffffffu, fi, l);
                        const float off = __shfl_sync(0xffffffffu, lrow - m, l);  // L_l - m_l
                        // exact term: log2(P/a_l) = log2 b_j + kappa (f_l + g_j - C_lj); the
                        // potentials and C_lj cancel to a small number: float-float throughout
                        const float2 pot = ff_add(two_sum(fl, gj), make_float2(-C2.x, -C2.y));
                        const float2 ell = ff_add(ff_mul(kap, pot), two_sum(lbj, off));
                        const float w = exp2f(__fadd_rn(ell.x, ell.y));
                        const float Cf = __fadd_rn(C2.x, C2.y);
                        if (lane == l) {
                            r += w - ex2f(e);
                            q = fmaf(w, Cf, q);
                        }
                        float* vr = x.vpart + (((size_t)ch * p.B * p.nr) + rbase + rl) * D + 2 * lane;
                        for (int sl = 0; sl < ns; ++sl) {
                            const float2 yv = *reinterpret_cast<const float2*>(yj + sl * TC_D);
                            float2 acc = *reinterpret_cast<float2*>(vr + sl * TC_D);
                            acc.x = fmaf(w, yv.x, acc.x);
                            acc.y = fmaf(w, yv.y, acc.y);
                            *reinterpret_cast<float2*>(vr + sl * TC_D) = acc;
                        }
                    }
                }
            }
            if (SL) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(S.bar(BAR_ACCEMPTY(wg, u)));
                    mbar_arrive(S.bar(BAR_BEMPTY(u)));
                }
            } else {
                tc_release(S, wg, lt);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (*abort) {
        m = NAN;
        if (threadIdx.x == 0) atomicOr(p.status, SOT_DEV_TIMEOUT);
    }
    const size_t stride = (size_t)p.B * p.nr;
    if (p.split > 1) {
        if (erow) {
            p.part_m[ch * stride + rbase + row] = m;
            x.part_r[ch * stride + rbase + row] = r;
            x.part_q[ch * stride + rbase + row] = q;
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = atomicAdd(&p.counters[b * p.rowtiles + rb], 1u);
            misc[3] = (prev == (unsigned)(p.split - 1));
        }
        __syncthreads();
        if (!misc[3]) return;
        __threadfence();
        if (threadIdx.x == 0) p.counters[b * p.rowtiles + rb] = 0u;
    }
    float qi = 0.f;
    if (erow) {
        // merge the chunks: scale each chunk's sums from its stabiliser to the largest
        float M = -INFINITY;
        bool nan = false;
        for (int c = 0; c < p.split; ++c) {
            const float mc = (p.split > 1) ? __ldcg(p.part_m + c * stride + rbase + row) : m;
            if (mc != mc) nan = true;
            M = fmaxf(M, mc);
        }
        float R = 0.f, Q = 0.f;
        for (int c = 0; c < p.split; ++c) {
            const float mc = (p.split > 1) ? __ldcg(p.part_m + c * stride + rbase + row) : m;
            const float f = (mc == -INFINITY || M == -INFINITY) ? 0.f : ex2f(mc - M);
            R += f * ((p.split > 1) ? __ldcg(x.part_r + c * stride + rbase + row) : r);
            Q += f * ((p.split > 1) ? __ldcg(x.part_q + c * stride + rbase + row) : q);
        }
        // the exponents were taken against m (= L_i - bias), so P_ij / a_i = 2^(e + m - L_i)
        const float ai = x.a ? x.a[rbase + row] : 1.f / (float)p.nr;
        const float fac = nan ? NAN : ai * ex2f(M - p.rstate_in[rbase + row]);
        const float ri = fac * R;
        qi = fac * Q;
        if (x.rowsum) x.rowsum[rbase + row] = ri;
        if (x.grad) {
            // v in caller coordinates, merged over the chunks 64 coordinates at a time
            for (int k0 = 0; k0 < D; k0 += TC_D) {
                float V[TC_D];
#pragma unroll
                for (int k = 0; k < TC_D; ++k) V[k] = 0.f;
                for (int c = 0; c < p.split; ++c) {
                    const float mc = (p.split > 1) ? __ldcg(p.part_m + c * stride + rbase + row) : m;
                    const float f = (mc == -INFINITY || M == -INFINITY) ? 0.f : ex2f(mc - M);
                    const float* vc = x.vpart + ((size_t)c * stride + rbase + row) * D + k0;
#pragma unroll
                    for (int k = 0; k < TC_D; ++k) V[k] = fmaf(f, __ldcg(vc + k), V[k]);
                }
                const float* xo = x.X + (rbase + row) * D + k0;
                float* gr = x.grad + (rbase + row) * D + k0;
#pragma unroll
                for (int k = 0; k < TC_D; ++k) gr[k] = 2.f * (ai * xo[k] - fac * V[k]);
            }
        }
    }
    if (x.cost_part) {
        qi = block_sum<TC_THREADS>(qi, red);
        if (threadIdx.x == 0) x.cost_part[b * p.rowtiles + rb] = qi;
    }
}

size_t tc_apply_scratch_floats(int B, int n, int d, int split) {
    return (size_t)split * B * n * (d + 2);
}

cudaError_t launch_tc_apply(const TcPlan& plan, const ApplyArgs& a, const HalfArgs& hp, float* scratch,
                            cudaStream_t st) {
    if (!tc_supported(a.d) || a.d != plan.d || plan.S != tc_slices(a.d)) return cudaErrorInvalidValue;
    TcOps ops;
    ops.aimg = plan.xop;
    ops.bimg = plan.yop;
    ops.scale = plan.scale;
    ops.tiles_r = plan.tiles_x;
    ops.tiles_c = plan.tiles_y;
    ops.S = plan.S;
    ops.bias = plan.bias;
    ops.bias_img = nullptr;
    tc_fill_waits(ops);
    {
        const cudaError_t eb = launch_tc_bias(plan, hp, ops.tiles_c, st);
        if (eb != cudaSuccess) return eb;
    }
    TcApplyExtra x;
    const size_t rows = (size_t)a.B * a.n;
    x.nx = a.nx;
    x.ny = a.ny;
    x.X = a.X;
    x.Y = a.Yorig;
    x.f = a.fpot;
    x.g = a.gpot;
    x.kappa64 = a.kappa64;
    x.a = a.a;
    x.shift = a.shift;
    x.vpart = scratch;
    x.part_r = scratch + (size_t)hp.split * rows * a.d;
    x.part_q = x.part_r + (size_t)hp.split * rows;
    x.cost_part = a.cost_part;
    x.grad = a.grad;
    x.rowsum = a.rowsum;
    cudaError_t e = cudaMemsetAsync(x.vpart, 0, sizeof(float) * (size_t)hp.split * rows * a.d, st);
    if (e != cudaSuccess) return e;
    dim3 grid(hp.rowtiles * hp.split, hp.B), block(TC_THREADS);
    if (plan.S == 1) {
        e = cudaFuncSetAttribute(tc_apply_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
        if (e != cudaSuccess) return e;
        count_launches(1);
        tc_apply_kernel<false><<<grid, block, TC_SMEM, st>>>(hp, ops, x);
    } else {
        e = cudaFuncSetAttribute(tc_apply_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
        if (e != cudaSuccess) return e;
        count_launches(1);
        tc_apply_kernel<true><<<grid, block, TC_SMEM, st>>>(hp, ops, x);
    }
    return cudaGetLastError();
}

}  // namespace sot
