// k_tc.cu -- tcgen05 tensor-core half-steps (placeholder: no tensor-core
// kernel is compiled in yet, so tc_supported() is false and every dimension
// takes the fp32 paths).
#include "tc.h"

namespace sot {

bool tc_supported(int) { return false; }
int tc_max_d() { return 0; }
int tc_rows_per_cta() { return 128; }
int tc_cols_per_tile() { return 128; }
size_t tc_scratch_bytes(int, int, int, int) { return 0; }
cudaError_t tc_prepare(TcPlan&, unsigned char*, int, int, int, int, const float*, const float*, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_tc_half(const TcPlan&, const HalfArgs&, int, int, cudaStream_t) { return cudaErrorNotSupported; }
bool tc_apply_supported(int) { return false; }
int tc_apply_rows_per_cta() { return 128; }
cudaError_t launch_tc_apply(const TcPlan&, const ApplyArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sot
