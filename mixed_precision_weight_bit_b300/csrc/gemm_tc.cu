// Tensor-core dequant-MMA for batches of 2..256 columns (not yet built for the current layout).
#include "internal.h"

namespace vbq {

bool tc_eligible(const vbq_matrix*) { return false; }
vbq_status launch_gemm_tc(const vbq_matrix*, const uint16_t*, int32_t, float*, cudaStream_t) {
  return fail(VBQ_ERR_UNSUPPORTED, "tensor-core path not built");
}
void tc_forget(const vbq_matrix*) {}

}  // namespace vbq
