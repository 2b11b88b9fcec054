// tc.h -- interface of the tcgen05 (5th-generation tensor core) Sinkhorn
// path, k_tc.cu.  Internal to libsot.
#pragma once
#include <cuda_runtime.h>

#include "kernels.h"

namespace sot {

// Operand images for the tensor-core half-steps, prepared once per call from
// the centred coordinates.
struct TcPlan {
    int B = 0, n = 0, m = 0, d = 0;
    int S = 1;                     // slices of K = 64 per image tile (d / 64)
    int tiles_x = 0, tiles_y = 0;  // 128-point tiles per cloud in each image (even count)
    unsigned char* xop = nullptr;  // operand image of X: per tile and slice 16 KB fp16 hi + 16 KB fp16 lo, swizzled
    unsigned char* yop = nullptr;  // operand image of Y
    float* scale = nullptr;        // [B] power-of-two coordinate scale used by the images
    float* bias = nullptr;         // [B][max tiles * 128] column biases of the current half-step
    unsigned* nrm = nullptr;       // [B][4] float bits: max |x hi|, max |x - x hi|, max |y hi|, max |y - y hi| (scaled)
    unsigned* cmax = nullptr;      // [3][B]: running max |c_j| (float bits), block counter, final max of the
                                   // last screened half-step's column biases; the first two zero between launches
    unsigned char* bimg = nullptr; // [B][max tiles] 16 KB tiles: fp16 parts of the column biases (screened)
};

// Screening state of the hi * hi half-step.  Every CTA appends the pairs it
// keeps to its own pool; the CTA that finishes a row block evaluates the
// pools of all its column chunks.
struct TcScreen {
    uint2* pool = nullptr;    // [B * rowtiles_max * split_max][pool_cap] (column, local row)
    int pool_cap = 0;
    int* pool_cnt = nullptr;  // [B * rowtiles_max * split_max][segments] entries used in each pool segment
    int* lost = nullptr;      // [B * max(n, m)] rows with a pair that did not fit; zero between launches
    int* ovf = nullptr;       // running count of lost rows
};

// Testing hook for the timeout path: after `after` more tensor-core launches,
// every tensor-core producer issues no copy from column tile `tile` of its
// chunk on (tile < 0: off), and every bounded wait gives up after wait_ns
// (0: 2 s).
void tc_set_test_hold(int tile, int after, unsigned long long wait_ns);
// The screened half-step takes d = 64, 128, 192, 256; the full half-step and
// the plan application d = 64 only.
bool tc_supported(int d);
bool tc_half_supported(int d);
int tc_max_d();
int tc_rows_per_cta();
int tc_cols_per_tile();
size_t tc_scratch_bytes(int B, int n, int m, int d);
cudaError_t tc_prepare(TcPlan& plan, unsigned char* scratch, int B, int n, int m, int d, const float* xc,
                       const float* yc, cudaStream_t st);
cudaError_t launch_tc_half(const TcPlan& plan, const HalfArgs& p, int h, int mode, cudaStream_t st);
// Screened half-step (warm half-steps only: needs p.lo_in): hi * hi products
// screen every pair against a bound of the row's new value; the candidates
// are evaluated exactly in fp32.  Same inputs and outputs as launch_tc_half.
cudaError_t launch_tc_screen(const TcPlan& plan, const HalfArgs& p, int h, const TcScreen& sc, cudaStream_t st);
int tc_screen_pool_cap();
int tc_screen_pool_segments();
bool tc_apply_supported(int d);
bool tc_apply_default();
int tc_apply_rows_per_cta();
// Plan application on the tensor cores.  `hp` carries the split plan and the
// f-half operands (rows X, columns Y, column state Lam, row state L); scratch
// holds tc_apply_scratch_floats() floats.
size_t tc_apply_scratch_floats(int B, int n, int d, int split);
cudaError_t launch_tc_apply(const TcPlan& plan, const ApplyArgs& a, const HalfArgs& hp, float* scratch,
                            cudaStream_t st);

}  // namespace sot
