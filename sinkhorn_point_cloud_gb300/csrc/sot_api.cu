// sot_api.cu -- the C ABI of libsot (declared in include/sot.h): argument
// checks, stream-ordered scratch, path choice, and the orchestration of the
// fused half-step kernels into fixed, annealed and stop-tested Sinkhorn
// solves ("FlashSinkhorn", Methodologie 1-3), plan application and the
// thresholded COO plan ("CUDA-Optimized APML", Abstract / Innovation).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "sot.h"
#include "apml.h"
#include "hvp.h"
#include "tc.h"
#include "transport.h"

using namespace sot;

namespace sot {
static std::atomic<long long> g_kernel_launches{0};
void count_launches(int k) { g_kernel_launches.fetch_add(k, std::memory_order_relaxed); }
long long launches_total() { return g_kernel_launches.load(std::memory_order_relaxed); }
}  // namespace sot

namespace {

constexpr double SOT_LN2_D = 0.69314718055994530942;

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

#define SOT_CUDA(call)                                                                   \
    do {                                                                                 \
        cudaError_t _e = (call);                                                         \
        if (_e != cudaSuccess)                                                           \
            return fail(SOT_ERR_CUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(_e), __FILE__, __LINE__); \
    } while (0)

// Bytes of freed scratch the library's pool keeps for later calls.
constexpr unsigned long long SCRATCH_KEEP_BYTES = 2ull << 30;

// One stream-ordered pool per device, owned by the library.  A device's
// default pool keeps no freed memory across a synchronisation, so every call
// would map its scratch afresh; this one keeps up to SCRATCH_KEEP_BYTES.
// NULL when the pool cannot be made (the caller then uses the default pool).
cudaMemPool_t scratch_pool() {
    static cudaMemPool_t pools[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps pr;
        std::memset(&pr, 0, sizeof(pr));
        pr.allocType = cudaMemAllocationTypePinned;
        pr.handleTypes = cudaMemHandleTypeNone;
        pr.location.type = cudaMemLocationTypeDevice;
        pr.location.id = dev;
        cudaMemPool_t mp = nullptr;
        if (cudaMemPoolCreate(&mp, &pr) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        unsigned long long keep = SCRATCH_KEEP_BYTES;
        if (cudaMemPoolSetAttribute(mp, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) cudaGetLastError();
        pools[dev] = mp;
    }
    return pools[dev];
}

// Stream-ordered scratch: every allocation is released on the same stream
// when the owning call returns.
struct Scratch {
    cudaStream_t st;
    std::vector<void*> ptrs;
    // Arena mode (sot_potentials_noalloc): carve 256-byte aligned pieces out of a
    // caller-provided device area instead of allocating; nothing is freed.
    unsigned char* arena = nullptr;
    size_t arena_cap = 0, arena_used = 0;
    explicit Scratch(cudaStream_t s) : st(s) {}
    Scratch(cudaStream_t s, unsigned char* base, size_t cap) : st(s), arena(base), arena_cap(cap) {}
    ~Scratch() {
        for (void* p : ptrs) cudaFreeAsync(p, st);
    }
    template <class T>
    T* alloc(size_t count) {
        void* p = nullptr;
        if (count == 0) count = 1;
        if (arena) {
            const size_t off = (arena_used + 255) & ~(size_t)255;
            if (off + count * sizeof(T) > arena_cap) return nullptr;
            arena_used = off + count * sizeof(T);
            return reinterpret_cast<T*>(arena + off);
        }
        cudaMemPool_t mp = scratch_pool();
        const cudaError_t e = mp ? cudaMallocFromPoolAsync(&p, count * sizeof(T), mp, st)
                                 : cudaMallocAsync(&p, count * sizeof(T), st);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        ptrs.push_back(p);
        return static_cast<T*>(p);
    }
};

// SM count of the current device, cached per device.  Concurrent first calls
// may both query; each stores the same value.  A failed query is not cached.
int device_sms() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 148;
    }
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 148;
    }
    cached[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ---- per-launch timing (sot_profile_*) ------------------------------------
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
    cudaEvent_t a, b;
    int kind;   // 0: full half-step, 1: screened half-step, 2: cluster-resident iterations
    int count;  // half-steps the timed launch(es) cover
};
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

struct ProfScope {
    cudaEvent_t a = nullptr, b = nullptr;
    cudaStream_t st;
    int kind = 0;
    int count = 1;
    ProfScope(cudaStream_t s, bool want) : st(s) {
        if (!want) return;
        std::lock_guard<std::mutex> g(g_prof_mu);
        if (!g_prof_on) return;
        a = prof_event();
        b = prof_event();
        cudaEventRecord(a, st);
    }
    ~ProfScope() {
        if (!a) return;
        cudaEventRecord(b, st);
        std::lock_guard<std::mutex> g(g_prof_mu);
        g_prof_pending.push_back(ProfRec{a, b, kind, count});
    }
};

enum Path { PATH_POINT = 0, PATH_DENSE = 1, PATH_TC = 2 };

// The tensor cores' dimension for d: the smallest of 64, 128, 192, 256, 512 and
// 1024 not below d (0 past 1024).  A cloud of another d runs there with its
// coordinates zero-padded.
int tc_dim(int d) {
    static const int dims[] = {64, 128, 192, 256, 512, 1024};
    for (int D : dims)
        if (d <= D) return D;
    return 0;
}
constexpr int TC_AUTO_MIN_D = 17;  // automatic precision takes the tensor cores above d = 16

int choose_path(int d, int flags, Path* out) {
    const int prec = flags & SOT_PREC_MASK;
    if (prec == SOT_PREC_F16X3) {
        if (d < 4 || !tc_dim(d))
            return fail(SOT_ERR_UNSUPPORTED, "SOT_PREC_F16X3 needs 4 <= d <= 1024 (got d = %d)", d);
        *out = PATH_TC;
        return SOT_OK;
    }
    if (prec != SOT_PREC_AUTO && prec != SOT_PREC_FP32) return fail(SOT_ERR_INVALID_ARG, "unknown precision flag");
    if (d <= 3) { *out = PATH_POINT; return SOT_OK; }
    if (prec == SOT_PREC_AUTO && d >= TC_AUTO_MIN_D && tc_dim(d)) { *out = PATH_TC; return SOT_OK; }
    if (d > dense_max_d()) return fail(SOT_ERR_UNSUPPORTED, "d = %d exceeds the fp32 path limit %d", d, dense_max_d());
    *out = PATH_DENSE;
    return SOT_OK;
}

int check_sizes(const float* X, const float* Y, int B, int n, int m, int d) {
    if (B < 0 || n <= 0 || m <= 0 || d <= 0)
        return fail(SOT_ERR_INVALID_ARG, "sizes must satisfy B >= 0, n, m, d >= 1 (got B=%d n=%d m=%d d=%d)", B, n, m, d);
    if (B > 65535) return fail(SOT_ERR_INVALID_ARG, "B = %d exceeds 65535", B);
    if ((long long)B * n * d >= (1LL << 40) || (long long)B * m * d >= (1LL << 40))
        return fail(SOT_ERR_INVALID_ARG, "problem too large");
    if ((long long)B * n >= (1LL << 31) || (long long)B * m >= (1LL << 31))
        return fail(SOT_ERR_INVALID_ARG, "B*n and B*m must be < 2^31");
    if (B > 0 && (!X || !Y)) return fail(SOT_ERR_INVALID_ARG, "X and Y must not be NULL");
    return SOT_OK;
}

// Cosine cost (SOT_COST_COSINE): unit copies of both clouds in `scr`, which
// stay alive (stream-ordered) for the rest of the call; *Xu, *Yu point at
// them.  Without the flag the inputs are used as they are.
int unit_points(int flags, const float* X, const float* Y, int B, int n, int m, int d, Scratch& scr,
                const float** Xu, const float** Yu) {
    *Xu = X;
    *Yu = Y;
    if (!(flags & SOT_COST_COSINE) || B == 0) return SOT_OK;
    float* xn = scr.alloc<float>((size_t)B * n * d);
    float* yn = scr.alloc<float>((size_t)B * m * d);
    if (!xn || !yn) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    SOT_CUDA(launch_normalise(X, (long long)B * n, d, xn, scr.st));
    SOT_CUDA(launch_normalise(Y, (long long)B * m, d, yn, scr.st));
    *Xu = xn;
    *Yu = yn;
    return SOT_OK;
}

// The tensor path at a d it does not take natively: zero-padded copies of both
// clouds at D = tc_dim(d) in `scr` (alive for the rest of the call).
int pad_points(const float* X, const float* Y, int B, int n, int m, int d, int D, Scratch& scr, const float** Xp,
               const float** Yp) {
    *Xp = X;
    *Yp = Y;
    if (D == d || B == 0) return SOT_OK;
    float* xp = scr.alloc<float>((size_t)B * n * D);
    float* yp = scr.alloc<float>((size_t)B * m * D);
    if (!xp || !yp) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    SOT_CUDA(launch_pad(X, (long long)B * n, d, D, xp, scr.st));
    SOT_CUDA(launch_pad(Y, (long long)B * m, d, D, yp, scr.st));
    *Xp = xp;
    *Yp = yp;
    return SOT_OK;
}

// Column split of one half-step: rows in tiles of rpc, columns in tiles of
// cpt; choose the number of column chunks that keeps the SMs busy (fewest
// "rounds" of resident CTAs per unit of work).
void choose_split(int B, int nr, int nc, int rpc, int cpt, int sms, int occ, int* split, int* chunk, int* rowtiles) {
    *rowtiles = (nr + rpc - 1) / rpc;
    const long long base = (long long)B * *rowtiles;
    const long long slots = (long long)sms * (occ > 0 ? occ : 1);
    const int ntiles = (nc + cpt - 1) / cpt;
    int smax = ntiles < 64 ? ntiles : 64;
    double best = 1e300;
    int bs = 1;
    for (int s = 1; s <= smax; ++s) {
        const long long units = base * s;
        const double rounds = (double)((units + slots - 1) / slots);
        const double t = rounds / s * (1.0 + 0.01 * (s - 1));
        if (t < best * 0.999) { best = t; bs = s; }
    }
    const int tiles_per_chunk = (ntiles + bs - 1) / bs;
    *chunk = tiles_per_chunk * cpt;
    *split = (nc + *chunk - 1) / *chunk;
}

// Annealing stages: eps_k = max(eps, eps_init * factor^k); the first k with
// eps_init * factor^k <= eps is the last (clamped) stage.
std::vector<float> stages_of(const sot_schedule& s) {
    std::vector<float> v;
    const double e_min = s.eps;
    if (!(s.eps_init > s.eps) || !(s.eps_factor > 0.f) || !(s.eps_factor < 1.f)) {
        v.push_back(s.eps);
        return v;
    }
    double e = s.eps_init;
    for (;;) {
        v.push_back((float)(e > e_min ? e : e_min));
        if (e <= e_min || v.size() > 100000) break;
        e *= (double)s.eps_factor;
    }
    return v;
}

// ---------------------------------------------------------------------------
struct Solver {
    int B, n, m, d;
    Path path;
    cudaStream_t st;
    const float *X, *Y, *a, *b;
    Scratch S;
    float *shift = nullptr, *xpack = nullptr, *ypack = nullptr, *lw2x = nullptr, *lw2y = nullptr;
    float *nx = nullptr, *ny = nullptr;
    float *L = nullptr, *Lnext = nullptr, *Lam = nullptr;
    float *part_m = nullptr, *part_s = nullptr, *errpart = nullptr, *err = nullptr;
    unsigned* counters = nullptr;
    int* dflags = nullptr;  // [0] status, [1] stop, [2] conv, [3..] per-stage iteration counts
    // Stabiliser bounds: lo[side][slot][B] = min over that side's rows of
    // (state before - state after) of its last half-steps (two slots, alternating).
    unsigned* lo = nullptr;
    int seq[2] = {0, 0};
    bool bound_ok = false;  // the other side's last bound is valid for the next half-step
    int nstage_slots = 0;
    int sms;
    int split[2], chunk[2], rowtiles[2];  // [0] f-half (rows X), [1] g-half (rows Y)
    int rpt[2] = {4, 4};                  // point path: rows per thread
    // Tensor path with d > 64: the screened half-step takes the warm half-steps,
    // the fp32 dense half-step (with its own split plan) every other one.
    bool tc_dense_full = false;
    int dsplit[2], dchunk[2], drowtiles[2];
    int last_rowtiles[2] = {0, 0};  // row tiles of the last half-step of each side (its error partials)
    TcPlan tc;
    // Screened tensor-core half-steps: allowed by the caller, and on for the
    // current stage until too many rows overflow their candidate lists.
    TcScreen scr;
    bool screen_allowed = false;
    bool screen_on = false;
    // The first screened iteration of a stage is on probation: a row block with
    // more overflowing rows than the kernel retries inline is left, unwritten,
    // to a full half-step launched right after (on the flagged blocks only).
    bool screen_probation = false;
    int* redo = nullptr;
    // Cluster-resident iterations (point path, clouds that fit in shared memory).
    bool cluster_allowed = false;
    bool cluster_ok = false;
    int cl_C = 0, cl_T = 0, cl_S = 0;
    size_t cl_smem = 0;

    Solver(const float* X_, const float* Y_, const float* a_, const float* b_, int B_, int n_, int m_, int d_, Path p,
           cudaStream_t s)
        : B(B_), n(n_), m(m_), d(d_), path(p), st(s), X(X_), Y(Y_), a(a_), b(b_), S(s) {
        sms = device_sms();
    }
    // Scratch carved from a fixed device area (no allocation).
    Solver(const float* X_, const float* Y_, const float* a_, const float* b_, int B_, int n_, int m_, int d_, Path p,
           cudaStream_t s, unsigned char* arena, size_t arena_cap)
        : B(B_), n(n_), m(m_), d(d_), path(p), st(s), X(X_), Y(Y_), a(a_), b(b_), S(s, arena, arena_cap) {
        sms = device_sms();
    }

    int prepare(int stage_slots) {
        nstage_slots = stage_slots;
        const bool point = (path == PATH_POINT);
        shift = S.alloc<float>((size_t)B * d);
        nx = S.alloc<float>((size_t)B * n);
        ny = S.alloc<float>((size_t)B * m);
        L = S.alloc<float>((size_t)B * n);
        Lam = S.alloc<float>((size_t)B * m);
        dflags = S.alloc<int>(3 + stage_slots);
        lo = S.alloc<unsigned>((size_t)4 * B);
        if (point) {
            xpack = S.alloc<float>((size_t)B * n * 4);
            ypack = S.alloc<float>((size_t)B * m * 4);
        } else {
            xpack = S.alloc<float>((size_t)B * n * d);
            ypack = S.alloc<float>((size_t)B * m * d);
            lw2x = S.alloc<float>((size_t)B * n);
            lw2y = S.alloc<float>((size_t)B * m);
        }
        if (!shift || !nx || !ny || !L || !Lam || !dflags || !lo || !xpack || !ypack || (!point && (!lw2x || !lw2y)))
            return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        SOT_CUDA(cudaMemsetAsync(dflags, 0, sizeof(int) * (3 + stage_slots), st));
        SOT_CUDA(cudaMemsetAsync(lo, 0xFF, sizeof(unsigned) * 4 * B, st));  // empty minima
        SOT_CUDA(launch_center(X, Y, B, n, m, d, shift, st));
        SOT_CUDA(launch_pack(X, a, B, n, d, shift, point, xpack, lw2x, nx, st));
        SOT_CUDA(launch_pack(Y, b, B, m, d, shift, point, ypack, lw2y, ny, st));
        // split plans for the two halves
        for (int h = 0; h < 2; ++h) {
            const int nr = h ? m : n, nc = h ? n : m;
            if (path == PATH_POINT)
                point_plan(B, nr, nc, sms, &rpt[h], &split[h], &chunk[h], &rowtiles[h]);
            else if (path == PATH_DENSE)
                choose_split(B, nr, nc, dense_rows_per_cta(), dense_cols_per_tile(), sms, 2, &split[h], &chunk[h],
                             &rowtiles[h]);
            else
                choose_split(B, nr, nc, tc_rows_per_cta(), tc_cols_per_tile(), sms, 1, &split[h], &chunk[h],
                             &rowtiles[h]);
        }
        tc_dense_full = (path == PATH_TC) && !tc_half_supported(d);
        for (int h = 0; h < 2; ++h) {
            dsplit[h] = split[h];
            dchunk[h] = chunk[h];
            drowtiles[h] = rowtiles[h];
            if (tc_dense_full)
                choose_split(B, h ? m : n, h ? n : m, dense_rows_per_cta(), dense_cols_per_tile(), sms, 2, &dsplit[h],
                             &dchunk[h], &drowtiles[h]);
        }
        if (point && cluster_allowed)
            cluster_ok = point_cluster_plan(B, n, m, sms, &cl_C, &cl_T, &cl_S, &cl_smem);
        const int smax = std::max(std::max(split[0], split[1]), std::max(dsplit[0], dsplit[1]));
        const size_t rows_max = (size_t)B * (n > m ? n : m);
        const int rt_max = std::max(std::max(rowtiles[0], rowtiles[1]), std::max(drowtiles[0], drowtiles[1]));
        if (smax > 1) {
            part_m = S.alloc<float>(rows_max * smax);
            part_s = S.alloc<float>(rows_max * smax);
            if (!part_m || !part_s) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        }
        counters = S.alloc<unsigned>((size_t)B * rt_max);
        errpart = S.alloc<float>((size_t)B * rt_max);
        err = S.alloc<float>((size_t)B);
        if (!counters || !errpart || !err) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        SOT_CUDA(cudaMemsetAsync(counters, 0, sizeof(unsigned) * B * rt_max, st));
        if (path == PATH_TC) {
            unsigned char* buf = S.alloc<unsigned char>(tc_scratch_bytes(B, n, m, d));
            if (!buf) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
            cudaError_t e = tc_prepare(tc, buf, B, n, m, d, xpack, ypack, st);
            if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "tensor-core operand preparation failed: %s", cudaGetErrorString(e));
            if (screen_allowed) {
                const size_t ctas0 = (size_t)rowtiles[0] * split[0], ctas1 = (size_t)rowtiles[1] * split[1];
                const size_t ctas = (size_t)B * (ctas0 > ctas1 ? ctas0 : ctas1);
                scr.pool_cap = tc_screen_pool_cap();
                scr.pool = S.alloc<uint2>(ctas * scr.pool_cap);
                scr.pool_cnt = S.alloc<int>(ctas * tc_screen_pool_segments());
                scr.lost = S.alloc<int>(rows_max);
                scr.ovf = S.alloc<int>(1);
                redo = S.alloc<int>((size_t)B * rt_max);
                if (!scr.pool || !scr.pool_cnt || !scr.lost || !scr.ovf || !redo)
                    return fail(SOT_ERR_NOMEM, "scratch allocation failed");
                SOT_CUDA(cudaMemsetAsync(scr.lost, 0, sizeof(int) * rows_max, st));
                SOT_CUDA(cudaMemsetAsync(scr.ovf, 0, sizeof(int), st));
            }
        } else {
            screen_allowed = false;
        }
        return SOT_OK;
    }

    int* stop_flag() { return dflags + 1; }
    int* conv_flag() { return dflags + 2; }

    // Arguments of one half-step.  h = 0: f-half (rows X, state L); h = 1: g-half (rows Y, state Lam).
    HalfArgs half_args(int h, float kappa, bool cold, const float* rin, float* rout, float* errp, bool guarded) {
        HalfArgs p;
        p.B = B;
        p.nr = h ? m : n;
        p.nc = h ? n : m;
        p.d = d;
        p.rpack = h ? ypack : xpack;
        p.cpack = h ? xpack : ypack;
        p.cw2 = h ? lw2x : lw2y;
        p.cstate = h ? L : Lam;
        p.rstate_in = rin;
        p.rstate_out = rout;
        p.rweight = h ? b : a;
        p.two_kappa = 2.f * kappa;
        p.cold = cold ? 1 : 0;
        p.split = split[h];
        p.chunk = chunk[h];
        p.rowtiles = rowtiles[h];
        p.rpt = rpt[h];
        p.part_m = part_m;
        p.part_s = part_s;
        p.counters = counters;
        p.errpart = errp;
        p.stop_flag = guarded ? stop_flag() : nullptr;
        p.status = dflags;
        p.redo = nullptr;
        return p;
    }

    // The same with the dense kernels' split plan (tensor path, d > 64).
    void use_dense_plan(HalfArgs& p, int h) const {
        p.split = dsplit[h];
        p.chunk = dchunk[h];
        p.rowtiles = drowtiles[h];
    }

    int half(int h, int mode, float kappa, bool cold, const float* rin, float* rout, float* errp, bool guarded) {
        HalfArgs p = half_args(h, kappa, cold, rin, rout, errp, guarded);
        p.lo_in = nullptr;
        p.lo_out = nullptr;
        p.lo_reset = nullptr;
        if (mode == MODE_LSE && lo) {
            p.lo_out = lo + (size_t)(2 * h + (seq[h] & 1)) * B;
            p.lo_reset = lo + (size_t)(2 * h + ((seq[h] + 1) & 1)) * B;
            if (!cold && bound_ok && seq[1 - h] > 0)
                p.lo_in = lo + (size_t)(2 * (1 - h) + ((seq[1 - h] - 1) & 1)) * B;
            ++seq[h];
        }
        cudaError_t e;
        {
            ProfScope ps(st, mode == MODE_LSE);
            if (path == PATH_POINT) {
                e = launch_point_half(p, mode, st);
            } else if (path == PATH_DENSE) {
                e = launch_dense_half(p, mode, st);
            } else if (mode == MODE_LSE && screen_on && !cold && p.lo_in) {
                ps.kind = 1;
                // On probation, row blocks with many overflowing rows are left to a full
                // tensor-core half-step launched right after.
                if (screen_probation && !tc_dense_full) {
                    SOT_CUDA(cudaMemsetAsync(redo, 0, sizeof(int) * (size_t)B * rowtiles[h], st));
                    p.redo = redo;
                }
                e = launch_tc_screen(tc, p, h, scr, st);
                if (e == cudaSuccess && p.redo) {
                    HalfArgs q = p;  // the flagged row blocks, in full (the bound slot is already reset)
                    q.lo_reset = nullptr;
                    e = launch_tc_half(tc, q, h, mode, st);
                }
            } else if (tc_dense_full) {
                use_dense_plan(p, h);
                e = launch_dense_half(p, mode, st);
            } else {
                e = launch_tc_half(tc, p, h, mode, st);
            }
        }
        last_rowtiles[h] = p.rowtiles;
        if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "half-step launch failed: %s", cudaGetErrorString(e));
        return SOT_OK;
    }

    int init_states(const float* f, const float* g, float kappa) {
        SOT_CUDA(launch_state_from_potential(nx, f, kappa, B * n, L, st));
        SOT_CUDA(launch_state_from_potential(ny, g, kappa, B * m, Lam, st));
        return SOT_OK;
    }

    int write_potentials(float* f, float* g, float kappa) {
        SOT_CUDA(launch_potential_from_state(nx, L, kappa, B * n, f, st));
        SOT_CUDA(launch_potential_from_state(ny, Lam, kappa, B * m, g, st));
        return SOT_OK;
    }

    // Plain iteration: f-half then g-half, both in place.  The first iteration
    // of a stage runs cold (stabiliser -inf); later ones use the bounds.
    int iterate(float kappa, bool cold, bool guarded) {
        int rc = half(0, MODE_LSE, kappa, cold, L, L, nullptr, guarded);
        if (rc) return rc;
        rc = half(1, MODE_LSE, kappa, cold, Lam, Lam, nullptr, guarded);
        bound_ok = true;
        return rc;
    }

    // `iters` warm iterations of the current stage in one cluster-resident
    // launch (after the stage's cold first iteration).  Sets *ran = false, and
    // changes nothing, when no cluster of the planned shape fits the device.
    int cluster_iterations(float kappa, long long iters, bool* ran) {
        *ran = false;
        if (!cluster_ok || iters < 1 || iters > (1 << 30)) return SOT_OK;
        cudaError_t e;
        {
            ProfScope ps(st, true);
            ps.kind = 2;
            ps.count = (int)(2 * iters);
            e = launch_point_cluster(B, n, m, xpack, ypack, L, Lam, 2.f * kappa, (int)iters, cl_C, cl_T, cl_S,
                                     cl_smem, st);
        }
        if (e == cudaErrorInvalidConfiguration) {
            (void)cudaGetLastError();
            cluster_ok = false;
            return SOT_OK;
        }
        if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "cluster launch failed: %s", cudaGetErrorString(e));
        bound_ok = false;  // the bounds of the streaming half-steps are stale now
        *ran = true;
        return SOT_OK;
    }

    // A new eps stage starts: states are rescaled, the last bounds no longer apply.
    void new_stage() {
        bound_ok = false;
        screen_on = screen_allowed;
        screen_probation = screen_allowed;
    }

    // After the first screened iteration of a stage: if more than 1 row in 200
    // (at least 16) had a kept pair that did not fit in its CTA's pool, the plan
    // is too dense at this eps for screening to pay, and the stage continues
    // with full half-steps.
    // Reads one device counter (a stream synchronisation).
    int screen_check() {
        screen_probation = false;
        if (!screen_on) return SOT_OK;
        int h = 0;
        SOT_CUDA(cudaMemcpyAsync(&h, scr.ovf, sizeof(int), cudaMemcpyDeviceToHost, st));
        SOT_CUDA(cudaStreamSynchronize(st));
        SOT_CUDA(cudaMemsetAsync(scr.ovf, 0, sizeof(int), st));
        const long long lim = (long long)B * (n + m) / 200;
        if (h > (lim > 16 ? lim : 16)) screen_on = false;
        return SOT_OK;
    }

    // Stop-tested step: the f-half of the next iteration evaluates the
    // row-marginal error of the current iterate; the decision either stops
    // (keeping the current iterate) or commits that f-half.
    int tested_fhalf(float kappa, float tol, int force) {
        if (!Lnext) {
            Lnext = S.alloc<float>((size_t)B * n);
            if (!Lnext) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        }
        int rc = half(0, MODE_LSE, kappa, !bound_ok, L, Lnext, errpart, true);
        if (rc) return rc;
        SOT_CUDA(launch_decide(errpart, B, last_rowtiles[0], tol, force, err, stop_flag(), conv_flag(), Lnext, L, B * n,
                               st));
        return SOT_OK;
    }
};

int read_flag(const int* dptr, cudaStream_t st, int* out) {
    SOT_CUDA(cudaMemcpyAsync(out, dptr, sizeof(int), cudaMemcpyDeviceToHost, st));
    SOT_CUDA(cudaStreamSynchronize(st));
    return SOT_OK;
}

int run_schedule(Solver& sv, const sot_schedule& s, const float* f0, const float* g0, float* f, float* g,
                 sot_stats* stt) {
    const std::vector<float> eps = stages_of(s);
    const int K = (int)eps.size();
    int rc = sv.prepare(K);
    if (rc) return rc;
    const bool warm = (s.flags & SOT_WARM_START) != 0;
    const bool early = (s.flags & SOT_STAGE_EARLY_EXIT) != 0;
    const bool testing = s.tol > 0.f;
    const int ips = s.iters_per_stage;
    const long long max_total = s.max_iters > 0 ? s.max_iters : (long long)ips * K;
    bool cold = !warm;
    {
        const float kappa0 = 1.f / (eps[0] * SOT_LN2_D);
        if (warm) {
            rc = sv.init_states(f0, g0, kappa0);
            if (rc) return rc;
        } else {
            // f = g = 0: the column state of the first f-half is Lam = kappa |y|^2
            SOT_CUDA(launch_state_cold(sv.nx, kappa0, sv.B * sv.n, sv.L, sv.st));
            SOT_CUDA(launch_state_cold(sv.ny, kappa0, sv.B * sv.m, sv.Lam, sv.st));
        }
    }
    std::vector<int> host_counts(K, -1);  // realised iterations of untested stages
    long long total = 0;                  // iterations realised so far
    int stages_done = 0;
    bool stopped_all = false;
    bool err_valid = false;
    for (int k = 0; k < K && !stopped_all; ++k) {
        if (total >= max_total) break;
        const float kappa = 1.f / (eps[k] * SOT_LN2_D);
        if (k > 0) {
            const float ratio = eps[k - 1] / eps[k];
            SOT_CUDA(launch_scale(sv.L, ratio, sv.B * sv.n, sv.st));
            SOT_CUDA(launch_scale(sv.Lam, ratio, sv.B * sv.m, sv.st));
        }
        SOT_CUDA(cudaMemsetAsync(sv.stop_flag(), 0, 2 * sizeof(int), sv.st));  // stop + conv
        sv.new_stage();
        cold = true;
        stages_done = k + 1;
        int* counter = sv.dflags + 3 + k;
        const bool final_stage = (k == K - 1);
        const bool test = testing && (early || final_stage);
        if (!test) {
            long long todo = ips;
            if (total + todo > max_total) todo = max_total - total;
            long long t0 = 0;
            if (sv.cluster_ok && todo >= 3) {
                // the cold first iteration streams; the rest run cluster-resident
                rc = sv.iterate(kappa, cold, false);
                if (rc) return rc;
                cold = false;
                bool ran = false;
                rc = sv.cluster_iterations(kappa, todo - 1, &ran);
                if (rc) return rc;
                t0 = ran ? todo : 1;
            }
            for (long long t = t0; t < todo; ++t) {
                rc = sv.iterate(kappa, cold, false);
                if (rc) return rc;
                cold = false;
                if (t == 1) {
                    rc = sv.screen_check();
                    if (rc) return rc;
                }
            }
            total += todo;
            host_counts[k] = (int)todo;
            continue;
        }
        // tested stage: first iteration plain, then tested iterations
        const long long stage_cap = final_stage ? (max_total - total) : (long long)ips;
        if (stage_cap <= 0) break;
        rc = sv.iterate(kappa, cold, false);
        if (rc) return rc;
        cold = false;
        SOT_CUDA(launch_count_iter(nullptr, counter, sv.st));
        long long enq = 1;
        const int chunk = 8;
        int stopped = 0;
        while (!stopped) {
            if (enq >= stage_cap) {
                if (final_stage) {
                    // evaluate the error of the returned iterate and stop
                    rc = sv.tested_fhalf(kappa, s.tol, 1);
                    if (rc) return rc;
                    err_valid = true;
                }
                break;
            }
            for (int c = 0; c < chunk && enq < stage_cap; ++c, ++enq) {
                rc = sv.tested_fhalf(kappa, s.tol, 0);
                if (rc) return rc;
                rc = sv.half(1, MODE_LSE, kappa, false, sv.Lam, sv.Lam, nullptr, true);
                if (rc) return rc;
                SOT_CUDA(launch_count_iter(sv.stop_flag(), counter, sv.st));
                if (enq == 1) {
                    rc = sv.screen_check();
                    if (rc) return rc;
                }
            }
            if (final_stage) {
                rc = read_flag(sv.stop_flag(), sv.st, &stopped);
                if (rc) return rc;
                if (stopped) err_valid = true;
            }
        }
        int realised = 0;
        rc = read_flag(counter, sv.st, &realised);
        if (rc) return rc;
        total += realised;
        if (final_stage) {
            int conv = 0;
            rc = read_flag(sv.conv_flag(), sv.st, &conv);
            if (rc) return rc;
            if (stt) stt->converged = conv;
            stopped_all = true;
        }
    }
    const float kappa_f = 1.f / (eps[stages_done > 0 ? stages_done - 1 : 0] * SOT_LN2_D);
    if (stt && !err_valid) {
        // evaluate the marginal error of the returned iterate without changing it
        SOT_CUDA(cudaMemsetAsync(sv.stop_flag(), 0, 2 * sizeof(int), sv.st));
        rc = sv.tested_fhalf(kappa_f, -1.f, 1);
        if (rc) return rc;
    }
    rc = sv.write_potentials(f, g, kappa_f);
    if (rc) return rc;
    if (stt) {
        std::vector<int> counts(K > 0 ? K : 1, 0);
        SOT_CUDA(cudaMemcpyAsync(counts.data(), sv.dflags + 3, sizeof(int) * K, cudaMemcpyDeviceToHost, sv.st));
        std::vector<float> errs(sv.B > 0 ? sv.B : 1, NAN);
        SOT_CUDA(cudaMemcpyAsync(errs.data(), sv.err, sizeof(float) * sv.B, cudaMemcpyDeviceToHost, sv.st));
        int dstatus = 0;
        SOT_CUDA(cudaMemcpyAsync(&dstatus, sv.dflags, sizeof(int), cudaMemcpyDeviceToHost, sv.st));
        SOT_CUDA(cudaStreamSynchronize(sv.st));
        if (dstatus & SOT_DEV_TIMEOUT)
            return fail(SOT_ERR_TIMEOUT, "a bounded device-side wait of a half-step gave up; the potentials are NaN");
        for (int k = 0; k < K; ++k)
            if (host_counts[k] >= 0) counts[k] = host_counts[k];
        long long tot = 0;
        for (int k = 0; k < stages_done; ++k) tot += counts[k];
        stt->iters_done = (int)tot;
        stt->stages_done = stages_done;
        if (!testing) stt->converged = 0;
        stt->final_eps = eps[stages_done > 0 ? stages_done - 1 : 0];
        if (stt->err_host)
            for (int i = 0; i < sv.B; ++i) stt->err_host[i] = errs[i];
        if (stt->stage_iters_host)
            for (int k = 0; k < stt->stage_iters_cap && k < K; ++k)
                stt->stage_iters_host[k] = k < stages_done ? counts[k] : 0;
    }
    return SOT_OK;
}

}  // namespace

// ===========================================================================
extern "C" {

int sot_version(void) { return 100; }

long long sot_kernel_launches(void) { return launches_total(); }

int sot_select_path(int d, int flags) {
    g_err[0] = 0;
    if (d <= 0) return fail(SOT_ERR_INVALID_ARG, "d must be >= 1");
    Path p;
    int rc = choose_path(d, flags, &p);
    return rc ? rc : (int)p;
}

const char* sot_last_error(void) { return g_err; }

const char* sot_status_string(int status) {
    switch (status) {
        case SOT_OK: return "ok";
        case SOT_ERR_INVALID_ARG: return "invalid argument";
        case SOT_ERR_NONFINITE: return "non-finite input or non-positive weight";
        case SOT_ERR_CAPACITY: return "COO capacity too small";
        case SOT_ERR_TIMEOUT: return "device wait timed out";
        case SOT_ERR_CUDA: return "CUDA error";
        case SOT_ERR_UNSUPPORTED: return "unsupported configuration";
        case SOT_ERR_NOMEM: return "out of device memory";
        default: return "unknown status";
    }
}

int sot_potentials_ex(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                      const sot_schedule* s, float* f, float* g, sot_stats* st, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!s) return fail(SOT_ERR_INVALID_ARG, "schedule must not be NULL");
    if (!(s->eps > 0.f) || !std::isfinite(s->eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (s->iters_per_stage < 0) return fail(SOT_ERR_INVALID_ARG, "iters_per_stage must be >= 0");
    if (s->flags & ~(SOT_PREC_MASK | SOT_WARM_START | SOT_STAGE_EARLY_EXIT | SOT_TC_NO_SCREEN | SOT_NO_CLUSTER |
                     SOT_COST_COSINE))
        return fail(SOT_ERR_INVALID_ARG, "unknown flag bits");
    if (B > 0 && (!f || !g)) return fail(SOT_ERR_INVALID_ARG, "f and g must not be NULL");
    if (st && st->stage_iters_host && st->stage_iters_cap < 0) return fail(SOT_ERR_INVALID_ARG, "stage_iters_cap < 0");
    if (B == 0) {
        if (st) { st->iters_done = 0; st->stages_done = 0; st->converged = 0; st->final_eps = s->eps; }
        return SOT_OK;
    }
    Path path;
    rc = choose_path(d, s->flags, &path);
    if (rc) return rc;
    // cosine cost: every step runs on the unit points
    Scratch unit((cudaStream_t)stream);
    rc = unit_points(s->flags, X, Y, B, n, m, d, unit, &X, &Y);
    if (rc) return rc;
    const int dr = (path == PATH_TC) ? tc_dim(d) : d;  // the dimension the kernels run at
    rc = pad_points(X, Y, B, n, m, d, dr, unit, &X, &Y);
    if (rc) return rc;
    Solver sv(X, Y, a, b, B, n, m, dr, path, (cudaStream_t)stream);
    sv.screen_allowed = (path == PATH_TC) && !(s->flags & SOT_TC_NO_SCREEN);
    sv.cluster_allowed = (path == PATH_POINT) && !(s->flags & SOT_NO_CLUSTER);
    rc = run_schedule(sv, *s, f, g, f, g, st);
    if (rc) return rc;
    if (!st) SOT_CUDA(launch_status_merge(sv.dflags, sv.st));  // asynchronous: reported by sot_async_status
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "%s", cudaGetErrorString(e));
    return SOT_OK;
}

int sot_async_status(void* stream) {
    g_err[0] = 0;
    unsigned v = 0;
    SOT_CUDA(read_clear_async_status((cudaStream_t)stream, &v));
    if (v & SOT_DEV_TIMEOUT)
        return fail(SOT_ERR_TIMEOUT, "a bounded device-side wait gave up in an asynchronous call; its rows are NaN");
    return SOT_OK;
}

int sot_test_hold_tile(int tile, int after_launches, long long wait_ns) {
    g_err[0] = 0;
    tc_set_test_hold(tile, after_launches, wait_ns > 0 ? (unsigned long long)wait_ns : 0ull);
    return SOT_OK;
}

int sot_potentials(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                   float eps, int iters, float* f, float* g, void* stream) {
    if (iters < 0) return fail(SOT_ERR_INVALID_ARG, "iters must be >= 0");
    sot_schedule s;
    s.eps = eps;
    s.eps_init = eps;
    s.eps_factor = 0.5f;
    s.iters_per_stage = iters;
    s.max_iters = iters;
    s.tol = 0.f;
    s.flags = 0;
    return sot_potentials_ex(X, Y, a, b, B, n, m, d, &s, f, g, nullptr, stream);
}

int sot_plan_apply(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                   const float* f, const float* g, float eps, float* cost, float* grad, float* rowsum, int flags,
                   void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (B > 0 && (!f || !g)) return fail(SOT_ERR_INVALID_ARG, "f and g must not be NULL");
    if (flags & ~(SOT_PREC_MASK | SOT_COST_COSINE)) return fail(SOT_ERR_INVALID_ARG, "unknown flag bits");
    if (B == 0 || (!cost && !grad && !rowsum)) return SOT_OK;
    const float* Xin = X;
    Scratch unit((cudaStream_t)stream);
    rc = unit_points(flags, X, Y, B, n, m, d, unit, &X, &Y);
    if (rc) return rc;
    Path path;
    rc = choose_path(d, flags, &path);
    if (rc) return rc;
    if (path == PATH_TC && (flags & SOT_PREC_MASK) == SOT_PREC_AUTO && !tc_apply_default()) path = PATH_DENSE;
    // Cosine cost: on unit points every score is below 2 kappa in magnitude, so
    // fp32 scores keep cost and gradient at fp32 accuracy, and the plan is often
    // dense (the tensor-core apply re-evaluates every significant pair exactly,
    // which only pays for a few pairs per row).
    if (path == PATH_TC && (flags & SOT_COST_COSINE) && (flags & SOT_PREC_MASK) == SOT_PREC_AUTO) path = PATH_DENSE;
    cudaStream_t cs = (cudaStream_t)stream;
    const int dr = (path == PATH_TC) ? tc_dim(d) : d;  // the dimension the kernels run at
    rc = pad_points(X, Y, B, n, m, d, dr, unit, &X, &Y);
    if (rc) return rc;
    float* gpad = nullptr;  // the gradient at dr, when that differs from d
    if (grad && dr != d) {
        gpad = unit.alloc<float>((size_t)B * n * dr);
        if (!gpad) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    }
    Solver sv(X, Y, a, b, B, n, m, dr, path, cs);
    rc = sv.prepare(0);
    if (rc) return rc;
    const float kappa = 1.f / (eps * SOT_LN2_D);
    rc = sv.init_states(f, g, kappa);
    if (rc) return rc;
    ApplyArgs p;
    p.B = B; p.n = n; p.m = m; p.d = dr;
    p.xpack = sv.xpack; p.ypack = sv.ypack; p.lw2x = sv.lw2x; p.lw2y = sv.lw2y;
    p.nx = sv.nx; p.ny = sv.ny; p.L = sv.L; p.Lam = sv.Lam;
    p.X = X; p.a = a; p.shift = sv.shift; p.kappa = kappa;
    p.Yorig = Y; p.fpot = f; p.gpot = g; p.kappa64 = 1.0 / ((double)eps * SOT_LN2_D);
    // above d = 256 the fp32 plan application takes the significant pairs' weights
    // exactly: the fp32 exponent's rounding, at the size of kappa |x||y|, grows with d
    p.exact_sig = (sv.path == PATH_DENSE && dr > 256) ? 1 : 0;
    const int rpc = (sv.path == PATH_POINT) ? point_apply_rows_per_cta()
                    : (sv.path == PATH_TC) ? tc_apply_rows_per_cta() : dense_apply_rows_per_cta();
    p.rowtiles = (sv.path == PATH_TC) ? sv.rowtiles[0] : (n + rpc - 1) / rpc;
    float* cpart = nullptr;
    if (cost) {
        cpart = sv.S.alloc<float>((size_t)B * p.rowtiles);
        if (!cpart) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    }
    p.cost_part = cpart; p.grad = gpad ? gpad : grad; p.rowsum = rowsum;
    cudaError_t e;
    if (sv.path == PATH_POINT) {
        e = launch_point_apply(p, cs);
    } else if (sv.path == PATH_TC) {
        float* scr = sv.S.alloc<float>(tc_apply_scratch_floats(B, n, dr, sv.split[0]));
        if (!scr) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        const HalfArgs hp = sv.half_args(0, kappa, false, sv.L, nullptr, nullptr, false);
        e = launch_tc_apply(sv.tc, p, hp, scr, cs);
    } else {
        e = launch_dense_apply(p, cs);
    }
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "plan-apply launch failed: %s", cudaGetErrorString(e));
    if (cost) SOT_CUDA(launch_reduce_parts(cpart, B, p.rowtiles, cost, cs));
    if (gpad)  // the first d coordinates of each row (the padded ones are zero)
        SOT_CUDA(cudaMemcpy2DAsync(grad, sizeof(float) * d, gpad, sizeof(float) * dr, sizeof(float) * d,
                                   (size_t)B * n, cudaMemcpyDeviceToDevice, cs));
    if (grad && (flags & SOT_COST_COSINE)) SOT_CUDA(launch_cosine_grad(Xin, (long long)B * n, d, grad, cs));
    SOT_CUDA(launch_status_merge(sv.dflags, cs));  // asynchronous: reported by sot_async_status
    return SOT_OK;
}

int sot_transport_apply(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                        const float* f, const float* g, float eps, const float* V, int c, int side, float* out,
                        int flags, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (side != 0 && side != 1) return fail(SOT_ERR_INVALID_ARG, "side must be 0 (P V) or 1 (P^T V), got %d", side);
    if (c < 1 || c > transport_max_c())
        return fail(SOT_ERR_INVALID_ARG, "c must satisfy 1 <= c <= %d (got %d)", transport_max_c(), c);
    if (d > transport_max_d())
        return fail(SOT_ERR_UNSUPPORTED, "transport products support d <= %d (got %d)", transport_max_d(), d);
    if (flags & ~SOT_COST_COSINE) return fail(SOT_ERR_INVALID_ARG, "unknown flag bits");
    if (B > 0 && (!f || !g || !V || !out)) return fail(SOT_ERR_INVALID_ARG, "f, g, V and out must not be NULL");
    if (B == 0) return SOT_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    Scratch unit(cs);
    rc = unit_points(flags, X, Y, B, n, m, d, unit, &X, &Y);
    if (rc) return rc;
    const double kap = 1.0 / ((double)eps * SOT_LN2_D);
    TransportArgs p;
    p.B = B; p.d = d; p.c = c; p.V = V; p.out = out; p.ldv = c; p.ldo = c;
    p.kap_hi = (float)kap;
    p.kap_lo = (float)(kap - (double)p.kap_hi);
    if (side == 0) {
        p.nr = n; p.nc = m; p.R = X; p.Cl = Y; p.fr = f; p.gc = g; p.wr = a; p.wc = b;
    } else {
        p.nr = m; p.nc = n; p.R = Y; p.Cl = X; p.fr = g; p.gc = f; p.wr = b; p.wc = a;
    }
    const size_t nparts = transport_plan(B, p.nr, p.nc, d, c, false, device_sms(), &p.split, &p.chunk);
    p.part = nparts ? unit.alloc<float>(nparts) : nullptr;
    if (nparts && !p.part) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    cudaError_t e = launch_transport(p, cs);
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "transport launch failed: %s", cudaGetErrorString(e));
    return SOT_OK;
}

int sot_grad_y(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
               const float* f, const float* g, float eps, float* grad_y, int flags, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (d > transport_max_d())
        return fail(SOT_ERR_UNSUPPORTED, "sot_grad_y supports d <= %d (got %d)", transport_max_d(), d);
    if (flags & ~SOT_COST_COSINE) return fail(SOT_ERR_INVALID_ARG, "unknown flag bits");
    if (B > 0 && (!f || !g || !grad_y)) return fail(SOT_ERR_INVALID_ARG, "f, g and grad_y must not be NULL");
    if (B == 0) return SOT_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const float* Yin = Y;
    Scratch unit(cs);
    rc = unit_points(flags, X, Y, B, n, m, d, unit, &X, &Y);
    if (rc) return rc;
    const double kap = 1.0 / ((double)eps * SOT_LN2_D);
    // P^T X, 64 coordinates of X per product, into grad_y
    for (int c0 = 0; c0 < d; c0 += transport_max_c()) {
        TransportArgs p;
        p.B = B; p.d = d; p.c = std::min(transport_max_c(), d - c0);
        p.nr = m; p.nc = n; p.R = Y; p.Cl = X; p.fr = g; p.gc = f; p.wr = b; p.wc = a;
        p.V = X + c0; p.ldv = d;
        p.out = grad_y + c0; p.ldo = d;
        p.kap_hi = (float)kap;
        p.kap_lo = (float)(kap - (double)p.kap_hi);
        const size_t nparts = transport_plan(B, p.nr, p.nc, d, p.c, false, device_sms(), &p.split, &p.chunk);
        p.part = nparts ? unit.alloc<float>(nparts) : nullptr;
        if (nparts && !p.part) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        cudaError_t e = launch_transport(p, cs);
        if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "transport launch failed: %s", cudaGetErrorString(e));
    }
    SOT_CUDA(launch_grad_finish(Y, b, B, m, d, grad_y, cs));
    if (flags & SOT_COST_COSINE) SOT_CUDA(launch_cosine_grad(Yin, (long long)B * m, d, grad_y, cs));
    return SOT_OK;
}

int sot_hvp(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
            const float* f, const float* g, float eps, const float* V, int cg_iters, float cg_tol, float* out,
            int flags, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (d > HVP_MAX_D) return fail(SOT_ERR_UNSUPPORTED, "sot_hvp supports d <= %d (got %d)", HVP_MAX_D, d);
    if (flags) return fail(SOT_ERR_INVALID_ARG, "sot_hvp takes no flags (squared-Euclidean cost only)");
    if (cg_iters < 1 || !(cg_tol >= 0.f) || !std::isfinite(cg_tol))
        return fail(SOT_ERR_INVALID_ARG, "cg_iters must be >= 1 and cg_tol finite and >= 0");
    if (B > 0 && (!f || !g || !V || !out)) return fail(SOT_ERR_INVALID_ARG, "f, g, V and out must not be NULL");
    if (B == 0) return SOT_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    const int c1 = 1 + d, c2 = 3 + d;
    const long long rn = (long long)B * n, rm = (long long)B * m;
    const double kap = 1.0 / ((double)eps * SOT_LN2_D);
    const int sms = device_sms();
    size_t nparts = 0;  // partial-sum scratch: the largest any of the products needs
    {
        int s, ch;
        nparts = std::max(nparts, transport_plan(B, n, m, d, c1, false, sms, &s, &ch));
        nparts = std::max(nparts, transport_plan(B, m, n, d, c2, false, sms, &s, &ch));
        nparts = std::max(nparts, transport_plan(B, n, m, d, 1, false, sms, &s, &ch));
        nparts = std::max(nparts, transport_plan(B, m, n, d, 1, false, sms, &s, &ch));
        nparts = std::max(nparts, transport_plan(B, n, m, d, 1, true, sms, &s, &ch));
    }
    Scratch S(cs);
    const size_t rmax = (size_t)B * std::max(n, m);
    float* shift = S.alloc<float>((size_t)B * d);
    float* Xc = S.alloc<float>((size_t)rn * d);
    float* Yc = S.alloc<float>((size_t)rm * d);
    float* lw = S.alloc<float>(rmax);
    float* nrm = S.alloc<float>(rmax);
    float* A1 = S.alloc<float>((size_t)rm * c1);
    float* PY1 = S.alloc<float>((size_t)rn * c1);
    float* W = S.alloc<float>((size_t)rn * c2);
    float* PT = S.alloc<float>((size_t)rm * c2);
    float* rhs = S.alloc<float>((size_t)rm);
    float* cvec = S.alloc<float>((size_t)rm);
    float* res = S.alloc<float>((size_t)rm);
    float* z = S.alloc<float>((size_t)rm);
    float* p = S.alloc<float>((size_t)rm);
    float* Sp = S.alloc<float>((size_t)rm);
    float* Ptq = S.alloc<float>((size_t)rm);
    float* gd = S.alloc<float>((size_t)rm);
    float* Pp = S.alloc<float>((size_t)rn);
    float* q = S.alloc<float>((size_t)rn);
    float* YH = S.alloc<float>((size_t)rn * d);
    float* CP = S.alloc<float>((size_t)rn * 2 * d);
    double* dd = S.alloc<double>((size_t)4 * B);
    float* part = nparts ? S.alloc<float>(nparts) : nullptr;
    if (!shift || !Xc || !Yc || !lw || !nrm || !A1 || !PY1 || !W || !PT || !rhs || !cvec || !res || !z || !p ||
        !Sp || !Ptq || !gd || !Pp || !q || !YH || !CP || !dd || (nparts && !part))
        return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    HvpDots dots{dd, dd + B, dd + 3 * B};
#define SOT_HVP_STEP(call)                                                                          \
    do {                                                                                            \
        cudaError_t _e = (call);                                                                    \
        if (_e != cudaSuccess) return fail(SOT_ERR_CUDA, "sot_hvp: %s", cudaGetErrorString(_e));    \
    } while (0)
    // Both clouds less their common centre t = (mean x + mean y) / 2: H does not
    // change under a common translation, and the right-hand side's terms
    // (r_i x_i - (P Y)_i, x_i . v_i - y_j . v_i) cancel at the size of |x|.
    SOT_HVP_STEP(launch_center(X, Y, B, n, m, d, shift, cs));
    SOT_HVP_STEP(launch_pack(X, a, B, n, d, shift, 0, Xc, lw, nrm, cs));
    SOT_HVP_STEP(launch_pack(Y, b, B, m, d, shift, 0, Yc, lw, nrm, cs));
    // side 0: o[B][n][c] = P Vin (Vin [B][m][c]); side 1: o[B][m][c] = P^T Vin (Vin [B][n][c])
    auto product = [&](int side, const float* Vin, int c, float* o) -> cudaError_t {
        TransportArgs t;
        t.B = B; t.d = d; t.c = c; t.V = Vin; t.out = o; t.ldv = c; t.ldo = c;
        t.kap_hi = (float)kap;
        t.kap_lo = (float)(kap - (double)t.kap_hi);
        if (side == 0) {
            t.nr = n; t.nc = m; t.R = Xc; t.Cl = Yc; t.fr = f; t.gc = g; t.wr = a; t.wc = b;
        } else {
            t.nr = m; t.nc = n; t.R = Yc; t.Cl = Xc; t.fr = g; t.gc = f; t.wr = b; t.wc = a;
        }
        transport_plan(B, t.nr, t.nc, d, c, false, sms, &t.split, &t.chunk);
        t.part = part;
        return launch_transport(t, cs);
    };
    // r and P Y, then the right-hand side of the marginal system and c
    SOT_HVP_STEP(launch_hvp_pack_ones(rm, d, Yc, A1, cs));
    SOT_HVP_STEP(product(0, A1, c1, PY1));
    SOT_HVP_STEP(launch_hvp_pack_side1(rn, d, Xc, V, PY1, W, cs));
    SOT_HVP_STEP(product(1, W, c2, PT));
    SOT_HVP_STEP(launch_hvp_rhs(rm, d, Yc, PT, rhs, cvec, cs));
    // conjugate gradients on S gdot = rhs, every cloud at once; every 8 steps
    // the host reads the clouds' residuals and stops when all are done
    SOT_HVP_STEP(launch_hvp_cg_init(B, m, rhs, cvec, res, z, p, gd, dots, cs));
    std::vector<double> hrz(2 * (size_t)B);
    for (int it = 0; it < cg_iters; ++it) {
        SOT_HVP_STEP(product(0, p, 1, Pp));
        SOT_HVP_STEP(launch_hvp_div_r(rn, d, Pp, PY1, q, cs));
        SOT_HVP_STEP(product(1, q, 1, Ptq));
        SOT_HVP_STEP(launch_hvp_cg_step(B, m, it, cg_tol, cvec, Ptq, p, Sp, res, z, gd, dots, cs));
        if ((it & 7) == 7 && it + 1 < cg_iters) {
            SOT_HVP_STEP(cudaMemcpyAsync(hrz.data(), dots.rz0, sizeof(double) * B, cudaMemcpyDeviceToHost, cs));
            SOT_HVP_STEP(cudaMemcpyAsync(hrz.data() + B, dots.rz + (size_t)((it + 1) & 1) * B, sizeof(double) * B,
                                         cudaMemcpyDeviceToHost, cs));
            SOT_HVP_STEP(cudaStreamSynchronize(cs));
            bool done = true;
            for (int k = 0; k < B; ++k)
                if (hrz[B + k] > (double)cg_tol * (double)cg_tol * hrz[k]) done = false;
            if (done) break;
        }
    }
    // assembly from the row-centred product of gdot: [sum_j P_ij ((y_j - yhat_i).v_i)(y_j - yhat_i),
    // sum_j P_ij gdot_j (y_j - yhat_i)]
    SOT_HVP_STEP(launch_hvp_barycentre(rn, d, PY1, YH, cs));
    {
        TransportArgs t;
        t.B = B; t.d = d; t.c = 1; t.V = gd; t.ldv = 1; t.out = CP; t.ldo = 2 * d;
        t.kap_hi = (float)kap;
        t.kap_lo = (float)(kap - (double)t.kap_hi);
        t.nr = n; t.nc = m; t.R = Xc; t.Cl = Yc; t.fr = f; t.gc = g; t.wr = a; t.wc = b;
        t.rc = YH; t.rv = V;
        transport_plan(B, n, m, d, 1, true, sms, &t.split, &t.chunk);
        t.part = part;
        SOT_HVP_STEP(launch_transport_centred(t, cs));
    }
    SOT_HVP_STEP(launch_hvp_assemble_centred(rn, d, eps, V, PY1, CP, out, cs));
#undef SOT_HVP_STEP
    return SOT_OK;
}

int sot_cost(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
             const float* f, const float* g, float eps, float* cost, void* stream) {
    if (B > 0 && !cost) return fail(SOT_ERR_INVALID_ARG, "cost must not be NULL");
    return sot_plan_apply(X, Y, a, b, B, n, m, d, f, g, eps, cost, nullptr, nullptr, 0, stream);
}
int sot_grad_x(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
               const float* f, const float* g, float eps, float* grad, void* stream) {
    if (B > 0 && !grad) return fail(SOT_ERR_INVALID_ARG, "grad must not be NULL");
    return sot_plan_apply(X, Y, a, b, B, n, m, d, f, g, eps, nullptr, grad, nullptr, 0, stream);
}
int sot_cost_grad(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                  const float* f, const float* g, float eps, float* cost, float* grad, void* stream) {
    if (B > 0 && (!cost || !grad)) return fail(SOT_ERR_INVALID_ARG, "cost and grad must not be NULL");
    return sot_plan_apply(X, Y, a, b, B, n, m, d, f, g, eps, cost, grad, nullptr, 0, stream);
}

namespace {
// Everything the COO passes read, prepared once: the solver's packed clouds and
// states for (f, g), and the row and column maxima of the two scores (computed
// by the maximum passes with the predicate's own fp32 chain).
struct CooPrep {
    Solver sv;
    CooArgs p;
    CooPrep(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
            cudaStream_t cs)
        : sv(X, Y, a, b, B, n, m, d, d <= 3 ? PATH_POINT : PATH_DENSE, cs) {}
    int run(const float* f, const float* g, float eps, float threshold, int dirs) {
        const int B = sv.B, n = sv.n, m = sv.m, d = sv.d;
        if (d > dense_max_d()) return fail(SOT_ERR_UNSUPPORTED, "COO extraction supports d <= %d", dense_max_d());
        int rc = sv.prepare(0);
        if (rc) return rc;
        const float kappa = 1.f / (eps * SOT_LN2_D);
        rc = sv.init_states(f, g, kappa);
        if (rc) return rc;
        float* Mr = sv.S.alloc<float>((size_t)B * n);
        float* Mc = sv.S.alloc<float>((size_t)B * m);
        int* counts = sv.S.alloc<int>((size_t)B * n);
        long long* rowptr = sv.S.alloc<long long>((size_t)B * n + 1);
        if (!Mr || !Mc || !counts || !rowptr) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
        rc = sv.half(0, MODE_MAX, kappa, true, nullptr, Mr, nullptr, false);
        if (rc) return rc;
        rc = sv.half(1, MODE_MAX, kappa, true, nullptr, Mc, nullptr, false);
        if (rc) return rc;
        p.B = B; p.n = n; p.m = m; p.d = d;
        p.xpack = sv.xpack; p.ypack = sv.ypack; p.lw2x = sv.lw2x; p.lw2y = sv.lw2y;
        p.nx = sv.nx; p.ny = sv.ny; p.L = sv.L; p.Lam = sv.Lam; p.Mr = Mr; p.Mc = Mc; p.a = sv.a;
        p.X = sv.X; p.Y = sv.Y; p.f = f; p.g = g;
        p.two_kappa = 2.f * kappa; p.kappa = kappa;
        const double kap = 1.0 / ((double)eps * SOT_LN2_D);
        p.kap_hi = (float)kap;
        p.kap_lo = (float)(kap - (double)p.kap_hi);
        p.log2tau = threshold > 0.f ? log2f(threshold) : -INFINITY;
        p.dirs = dirs;
        p.counts = counts; p.rowptr = rowptr; p.rows = nullptr; p.cols = nullptr; p.vals = nullptr;
        p.capacity = 0;
        return SOT_OK;
    }
};

int check_coo_args(float eps, float threshold, int dirs) {
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (!(threshold >= 0.f && threshold <= 1.f)) return fail(SOT_ERR_INVALID_ARG, "threshold must lie in [0, 1]");
    if (dirs < 1 || dirs > 3) return fail(SOT_ERR_INVALID_ARG, "dirs must be 1, 2 or 3");
    return SOT_OK;
}
}  // namespace

int sot_plan_coo(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                 const float* f, const float* g, float eps, float threshold, int dirs, long long capacity, int* rows,
                 int* cols, float* vals, long long* batch_offsets, long long* nnz_host, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!nnz_host) return fail(SOT_ERR_INVALID_ARG, "nnz_host must not be NULL");
    *nnz_host = 0;
    rc = check_coo_args(eps, threshold, dirs);
    if (rc) return rc;
    if (capacity < 0) return fail(SOT_ERR_INVALID_ARG, "capacity must be >= 0");
    if (B > 0 && (!f || !g || !batch_offsets)) return fail(SOT_ERR_INVALID_ARG, "f, g, batch_offsets must not be NULL");
    if (B == 0) return SOT_OK;
    if (capacity > 0 && (!rows || !cols || !vals)) return fail(SOT_ERR_INVALID_ARG, "rows, cols, vals must not be NULL");
    cudaStream_t cs = (cudaStream_t)stream;
    CooPrep cp(X, Y, a, b, B, n, m, d, cs);
    rc = cp.run(f, g, eps, threshold, dirs);
    if (rc) return rc;
    CooArgs& p = cp.p;
    p.rows = rows; p.cols = cols; p.vals = vals;
    p.capacity = capacity;
    cudaError_t e = (d <= 3) ? launch_point_coo(p, 0, cs) : launch_dense_coo(p, 0, cs);
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "COO count launch failed: %s", cudaGetErrorString(e));
    long long* rowptr = const_cast<long long*>(p.rowptr);
    SOT_CUDA(launch_scan_counts(p.counts, B, n, rowptr, batch_offsets, cs));
    long long nnz = 0;
    SOT_CUDA(cudaMemcpyAsync(&nnz, rowptr + (size_t)B * n, sizeof(long long), cudaMemcpyDeviceToHost, cs));
    SOT_CUDA(cudaStreamSynchronize(cs));
    *nnz_host = nnz;
    if (nnz > capacity) return fail(SOT_ERR_CAPACITY, "COO needs %lld entries, capacity %lld", nnz, capacity);
    if (nnz > 0) {
        e = (d <= 3) ? launch_point_coo(p, 1, cs) : launch_dense_coo(p, 1, cs);
        if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "COO write launch failed: %s", cudaGetErrorString(e));
    }
    return SOT_OK;
}

int sot_plan_coo_operands(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                          const float* f, const float* g, float eps, float threshold, float* xc, float* lwx, float* Lx,
                          float* yc, float* lwy, float* Ly, float* Mr, float* Mc, float* scalars_host, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    rc = check_coo_args(eps, threshold, 3);
    if (rc) return rc;
    if (!scalars_host) return fail(SOT_ERR_INVALID_ARG, "scalars_host must not be NULL");
    if (B == 0) return SOT_OK;
    if (!f || !g || !xc || !lwx || !Lx || !yc || !lwy || !Ly || !Mr || !Mc)
        return fail(SOT_ERR_INVALID_ARG, "f, g and every output must not be NULL");
    cudaStream_t cs = (cudaStream_t)stream;
    CooPrep cp(X, Y, a, b, B, n, m, d, cs);
    rc = cp.run(f, g, eps, threshold, 3);
    if (rc) return rc;
    const CooArgs& p = cp.p;
    const size_t fs = sizeof(float);
    for (int side = 0; side < 2; ++side) {
        const size_t cnt = (size_t)B * (side ? m : n);
        const float* pack = side ? p.ypack : p.xpack;
        float* oc = side ? yc : xc;
        float* ow = side ? lwy : lwx;
        if (d <= 3) {  // float4 (coordinates, log2 w) per point
            SOT_CUDA(cudaMemcpy2DAsync(oc, d * fs, pack, 4 * fs, d * fs, cnt, cudaMemcpyDeviceToDevice, cs));
            SOT_CUDA(cudaMemcpy2DAsync(ow, fs, pack + 3, 4 * fs, fs, cnt, cudaMemcpyDeviceToDevice, cs));
        } else {
            SOT_CUDA(cudaMemcpyAsync(oc, pack, cnt * d * fs, cudaMemcpyDeviceToDevice, cs));
            SOT_CUDA(cudaMemcpyAsync(ow, side ? p.lw2y : p.lw2x, cnt * fs, cudaMemcpyDeviceToDevice, cs));
        }
        SOT_CUDA(cudaMemcpyAsync(side ? Ly : Lx, side ? p.Lam : p.L, cnt * fs, cudaMemcpyDeviceToDevice, cs));
        SOT_CUDA(cudaMemcpyAsync(side ? Mc : Mr, side ? p.Mc : p.Mr, cnt * fs, cudaMemcpyDeviceToDevice, cs));
    }
    scalars_host[0] = p.kappa;
    scalars_host[1] = p.log2tau;
    return SOT_OK;
}

int sot_grad_x_coo(const float* X, const float* Y, int B, int n, int m, int d, const int* rows, const int* cols,
                   const float* vals, const long long* batch_offsets, float* grad, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (B == 0) return SOT_OK;
    if (!batch_offsets || !grad) return fail(SOT_ERR_INVALID_ARG, "batch_offsets and grad must not be NULL");
    cudaStream_t cs = (cudaStream_t)stream;
    Scratch S(cs);
    int* status = S.alloc<int>(1);
    if (!status) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    SOT_CUDA(cudaMemsetAsync(status, 0, sizeof(int), cs));
    SOT_CUDA(launch_grad_coo(X, Y, B, n, m, d, rows, cols, vals, batch_offsets, grad, status, cs));
    int h = 0;
    SOT_CUDA(cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, cs));
    SOT_CUDA(cudaStreamSynchronize(cs));
    if (h & SOT_DEV_BAD_COO) return fail(SOT_ERR_INVALID_ARG, "COO not row-sorted within a cloud or index out of range");
    return SOT_OK;
}

int sot_apml_coo(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                 const int* rows, const int* cols, const long long* batch_offsets, long long nnz, float T, int iters,
                 float* vals, float* loss, float* grad, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(T > 0.f) || !std::isfinite(T)) return fail(SOT_ERR_INVALID_ARG, "T must be finite and > 0");
    if (iters < 0) return fail(SOT_ERR_INVALID_ARG, "iters must be >= 0");
    if (nnz < 0 || nnz >= (1LL << 31)) return fail(SOT_ERR_INVALID_ARG, "nnz must satisfy 0 <= nnz < 2^31");
    if (B == 0) return SOT_OK;
    if (!batch_offsets || (nnz > 0 && (!rows || !cols || !vals)))
        return fail(SOT_ERR_INVALID_ARG, "batch_offsets, rows, cols and vals must not be NULL");
    cudaStream_t cs = (cudaStream_t)stream;
    ApmlArgs p;
    p.B = B; p.n = n; p.m = m; p.d = d;
    p.X = X; p.Y = Y; p.a = a; p.b = b;
    p.rows = rows; p.cols = cols; p.off = batch_offsets; p.nnz = nnz;
    p.inv_T = 1.f / T;
    p.iters = iters;
    p.vals = vals;
    p.loss = loss;
    p.grad = d <= 3 ? grad : nullptr;  // fused into the last pass
    const size_t nparts = apml_plan(B, n, m, device_sms(), &p.cpc, &p.rpc);
    const size_t bn = (size_t)B * n, bm = (size_t)B * m;
    // one scratch block, carved in 256-byte aligned pieces
    size_t total = 0;
    auto piece = [&](size_t bytes) {
        const size_t o = total;
        total += (std::max<size_t>(bytes, 1) + 255) & ~(size_t)255;
        return o;
    };
    const size_t o_cost = piece(sizeof(float) * (size_t)nnz), o_rs = piece(sizeof(int) * bn),
                 o_re = piece(sizeof(int) * bn), o_rstat = piece(sizeof(float2) * bn), o_uf = piece(sizeof(float) * bn),
                 o_cm = piece(sizeof(float) * bm), o_cf = piece(sizeof(float) * bm), o_vf = piece(sizeof(float) * bm),
                 o_part = piece(sizeof(float) * nparts), o_cmax = piece(nparts ? 0 : sizeof(unsigned) * bm),
                 o_csum = piece(nparts ? 0 : sizeof(double) * bm), o_lp = piece(sizeof(float) * bn),
                 o_st = piece(sizeof(int));
    Scratch S(cs);
    unsigned char* blk = S.alloc<unsigned char>(total);
    if (!blk) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    p.cost = reinterpret_cast<float*>(blk + o_cost);
    p.rstart = reinterpret_cast<int*>(blk + o_rs);
    p.rend = reinterpret_cast<int*>(blk + o_re);
    p.rstat = reinterpret_cast<float2*>(blk + o_rstat);
    p.ufac = reinterpret_cast<float*>(blk + o_uf);
    p.cm = reinterpret_cast<float*>(blk + o_cm);
    p.cfac = reinterpret_cast<float*>(blk + o_cf);
    p.vfac = reinterpret_cast<float*>(blk + o_vf);
    p.part = nparts ? reinterpret_cast<float*>(blk + o_part) : nullptr;
    p.cmax = nparts ? nullptr : reinterpret_cast<unsigned*>(blk + o_cmax);
    p.csum = nparts ? nullptr : reinterpret_cast<double*>(blk + o_csum);
    p.loss_part = reinterpret_cast<float*>(blk + o_lp);
    p.status = reinterpret_cast<int*>(blk + o_st);
    // rstart and rend are adjacent pieces: one clear covers both
    SOT_CUDA(cudaMemsetAsync(p.rstart, 0, o_rstat - o_rs, cs));
    if (!nparts) SOT_CUDA(cudaMemsetAsync(blk + o_cmax, 0, o_lp - o_cmax, cs));
    SOT_CUDA(cudaMemsetAsync(p.status, 0, sizeof(int), cs));
    // the offsets are checked on the device by the first pass, which bounds every
    // index the later passes take
    cudaError_t e = launch_apml(p, cs);
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "APML launch failed: %s", cudaGetErrorString(e));
    const char* bad = "batch_offsets not non-decreasing from 0 to nnz, COO not row-sorted within a cloud, or index "
                      "out of range";
    int h = 0;
    SOT_CUDA(cudaMemcpyAsync(&h, p.status, sizeof(int), cudaMemcpyDeviceToHost, cs));
    SOT_CUDA(cudaStreamSynchronize(cs));
    if (h & SOT_DEV_BAD_COO) return fail(SOT_ERR_INVALID_ARG, "%s", bad);
    if (grad && !p.grad) {  // d > 3: the gradient's own pass, on offsets now known to be valid
        SOT_CUDA(launch_grad_coo(X, Y, B, n, m, d, rows, cols, vals, batch_offsets, grad, p.status, cs));
        SOT_CUDA(cudaMemcpyAsync(&h, p.status, sizeof(int), cudaMemcpyDeviceToHost, cs));
        SOT_CUDA(cudaStreamSynchronize(cs));
        if (h & SOT_DEV_BAD_COO) return fail(SOT_ERR_INVALID_ARG, "%s", bad);
    }
    return SOT_OK;
}

int sot_check_inputs(const float* X, const float* Y, const float* a, const float* b, int B, int n, int m, int d,
                     void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (B == 0) return SOT_OK;
    cudaStream_t cs = (cudaStream_t)stream;
    Scratch S(cs);
    int* bad = S.alloc<int>(1);
    if (!bad) return fail(SOT_ERR_NOMEM, "scratch allocation failed");
    SOT_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), cs));
    SOT_CUDA(launch_check_inputs(X, a, (long long)B * n, d, (long long)B * n, bad, cs));
    SOT_CUDA(launch_check_inputs(Y, b, (long long)B * m, d, (long long)B * m, bad, cs));
    int h = 0;
    SOT_CUDA(cudaMemcpyAsync(&h, bad, sizeof(int), cudaMemcpyDeviceToHost, cs));
    SOT_CUDA(cudaStreamSynchronize(cs));
    if (h) return fail(SOT_ERR_NONFINITE, "%s", (h & 1) ? "non-finite coordinate" : "weight not finite or <= 0");
    return SOT_OK;
}

int sot_profile_enable(int on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_prof_on = on != 0;
    return SOT_OK;
}

int sot_profile_read_kinds(long long* launches_host, double* ms_host) {
    std::vector<ProfRec> pend;
    {
        std::lock_guard<std::mutex> g(g_prof_mu);
        pend.swap(g_prof_pending);
    }
    long long cnt[3] = {0, 0, 0};
    double ms[3] = {0.0, 0.0, 0.0};
    int rc = SOT_OK;
    for (auto& pr : pend) {
        float t = 0.f;
        if (rc == SOT_OK && cudaEventSynchronize(pr.b) != cudaSuccess) rc = fail(SOT_ERR_CUDA, "event synchronisation failed");
        if (rc == SOT_OK && cudaEventElapsedTime(&t, pr.a, pr.b) != cudaSuccess) rc = fail(SOT_ERR_CUDA, "event timing failed");
        cnt[pr.kind] += pr.count;
        ms[pr.kind] += t;
    }
    {
        std::lock_guard<std::mutex> g(g_prof_mu);
        for (auto& pr : pend) {
            g_prof_pool.push_back(pr.a);
            g_prof_pool.push_back(pr.b);
        }
    }
    if (rc) return rc;
    for (int k = 0; k < 3; ++k) {
        if (launches_host) launches_host[k] = cnt[k];
        if (ms_host) ms_host[k] = ms[k];
    }
    return SOT_OK;
}

int sot_profile_read(long long* launches_host, double* total_ms_host) {
    long long c[3];
    double t[3];
    const int rc = sot_profile_read_kinds(c, t);
    if (rc) return rc;
    if (launches_host) *launches_host = c[0] + c[1] + c[2];
    if (total_ms_host) *total_ms_host = t[0] + t[1] + t[2];
    return SOT_OK;
}

}  // extern "C"

// ===========================================================================
// Potentials without any allocation (sot_potentials_noalloc in sot.h).
//
// The scratch of the point-cloud solve lives in one statically sized device
// array that every GPU loading this library holds until the process exits.
// Host code must not use the array's name as a device address (on the host it
// is only a stand-in): the address is obtained once per device with
// cudaGetSymbolAddress and passed to the kernels.
static __device__ __align__(256) unsigned char g_sot_noalloc_scratch[SOT_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {nullptr};

// Device address of the static scratch on the current device (looked up on the
// first call for that device, with that device current).
int noalloc_scratch(unsigned char** out) {
    int dev = 0;
    SOT_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(SOT_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_sot_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(SOT_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
        g_noalloc_addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_noalloc_addr[dev]);
    return SOT_OK;
}

// Bytes the point-path solve carves from the arena (mirrors Solver::prepare
// for the point layout with no stage slots; 256-byte aligned pieces).
size_t noalloc_required_bytes(int B, int n, int m, int d) {
    auto piece = [](size_t bytes) { return ((bytes ? bytes : 1) + 255) & ~(size_t)255; };
    const size_t Bn = (size_t)B * n, Bm = (size_t)B * m;
    size_t total = piece(sizeof(float) * B * d) + piece(4 * Bn) + piece(4 * Bm) + piece(4 * Bn) + piece(4 * Bm) +
                   piece(sizeof(int) * 3) + piece(sizeof(unsigned) * 4 * B) + piece(16 * Bn) + piece(16 * Bm);
    int split[2], chunk[2], rowtiles[2], rpt[2];
    const int sms = device_sms();
    for (int h = 0; h < 2; ++h) point_plan(B, h ? m : n, h ? n : m, sms, &rpt[h], &split[h], &chunk[h], &rowtiles[h]);
    const int smax = split[0] > split[1] ? split[0] : split[1];
    const int rt_max = rowtiles[0] > rowtiles[1] ? rowtiles[0] : rowtiles[1];
    const size_t rows_max = (size_t)B * (n > m ? n : m);
    if (smax > 1) total += 2 * piece(4 * rows_max * smax);
    total += piece(4 * (size_t)B * rt_max) * 2 + piece(4 * (size_t)B);
    return total;
}

}  // namespace

extern "C" int sot_potentials_noalloc(const float* X, const float* Y, const float* a, const float* b, int B, int n,
                                      int m, int d, float eps, int iters, float* f, float* g, void* stream) {
    g_err[0] = 0;
    int rc = check_sizes(X, Y, B, n, m, d);
    if (rc) return rc;
    if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SOT_ERR_INVALID_ARG, "eps must be finite and > 0");
    if (iters < 0) return fail(SOT_ERR_INVALID_ARG, "iters must be >= 0");
    if (d > 3) return fail(SOT_ERR_UNSUPPORTED, "sot_potentials_noalloc serves point clouds with d <= 3 (got d = %d)", d);
    if (B == 0) return SOT_OK;
    if (!f || !g) return fail(SOT_ERR_INVALID_ARG, "f and g must not be NULL");
    const size_t need = noalloc_required_bytes(B, n, m, d);
    if (need > (size_t)SOT_NOALLOC_SCRATCH_BYTES)
        return fail(SOT_ERR_INVALID_ARG,
                    "B=%d n=%d m=%d needs %zu bytes of scratch; the static area holds %zu bytes "
                    "(use sot_potentials for larger problems)",
                    B, n, m, need, (size_t)SOT_NOALLOC_SCRATCH_BYTES);
    unsigned char* base = nullptr;
    rc = noalloc_scratch(&base);
    if (rc) return rc;
    cudaStream_t cs = (cudaStream_t)stream;
    Solver sv(X, Y, a, b, B, n, m, d, PATH_POINT, cs, base, (size_t)SOT_NOALLOC_SCRATCH_BYTES);
    rc = sv.prepare(0);  // zeroes the flags, bounds and merge counters left by the previous call
    if (rc) return rc;
    const float kappa = 1.f / (eps * SOT_LN2_D);
    SOT_CUDA(launch_state_cold(sv.nx, kappa, B * n, sv.L, cs));
    SOT_CUDA(launch_state_cold(sv.ny, kappa, B * m, sv.Lam, cs));
    for (int t = 0; t < iters; ++t) {
        rc = sv.iterate(kappa, t == 0, false);
        if (rc) return rc;
    }
    rc = sv.write_potentials(f, g, kappa);
    if (rc) return rc;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SOT_ERR_CUDA, "%s", cudaGetErrorString(e));
    return SOT_OK;
}
