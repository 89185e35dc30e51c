// Launch helpers shared by the API translation units.
#pragma once

#include <cuda_runtime.h>

#include "gemv.cuh"
#include "internal.h"

namespace vbq {

MatView view_of(const vbq_matrix* m, float* y, int32_t y_ld, float* trace_y);

// Sets kernel attributes and caches occupancy for nb columns. Call outside stream capture.
void warm_gemv(int nb);

// Launches the fused GEMV for nb in {1,2,4,8} batch columns over total_tiles
// tiles (summed over the segments of a). force_cluster > 0 fixes the cluster
// size; otherwise it is the largest of 8/4/2/1 that keeps one wave.
cudaError_t launch_gemv(int nb, const GemvArgs& a, int total_tiles, cudaStream_t st, bool pdl, int force_cluster);

}  // namespace vbq
