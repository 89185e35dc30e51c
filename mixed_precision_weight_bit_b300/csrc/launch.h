// Launch helpers shared by the API translation units.
#pragma once

#include <cuda_runtime.h>

#include "gemv.cuh"
#include "internal.h"

namespace vbq {

MatView view_of(const vbq_matrix* m, float* y, int32_t y_ld, float* trace_y);
PlanView plan_view(const DevicePlan& p);

// Sets the kernel attributes for nb batch columns. Call outside stream capture.
void warm_gemv(int nb);

// Launches the fused GEMV for nb in {1, 2, 4} batch columns with one CTA per
// entry of the plan (n_ctas). pdl lets the launch overlap the previous kernel.
cudaError_t launch_gemv(int nb, const GemvArgs& a, int n_ctas, cudaStream_t st, bool pdl);

}  // namespace vbq
