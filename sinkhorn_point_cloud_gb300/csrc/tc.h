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
    int tiles_x = 0, tiles_y = 0;  // 128-point tiles per cloud in each image (even count)
    unsigned char* xop = nullptr;  // operand image of X: per tile 16 KB fp16 hi + 16 KB fp16 lo, swizzled
    unsigned char* yop = nullptr;  // operand image of Y
    float* scale = nullptr;        // [B] power-of-two coordinate scale used by the images
};

bool tc_supported(int d);
int tc_max_d();
int tc_rows_per_cta();
int tc_cols_per_tile();
size_t tc_scratch_bytes(int B, int n, int m, int d);
cudaError_t tc_prepare(TcPlan& plan, unsigned char* scratch, int B, int n, int m, int d, const float* xc,
                       const float* yc, cudaStream_t st);
cudaError_t launch_tc_half(const TcPlan& plan, const HalfArgs& p, int h, int mode, cudaStream_t st);
bool tc_apply_supported(int d);
bool tc_apply_default();
int tc_apply_rows_per_cta();
// Plan application on the tensor cores.  `hp` carries the split plan and the
// f-half operands (rows X, columns Y, column state Lam, row state L); scratch
// holds tc_apply_scratch_floats() floats.
size_t tc_apply_scratch_floats(int B, int n, int split);
cudaError_t launch_tc_apply(const TcPlan& plan, const ApplyArgs& a, const HalfArgs& hp, float* scratch,
                            cudaStream_t st);

}  // namespace sot
