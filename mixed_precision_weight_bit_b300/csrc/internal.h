// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/vbq.h"
#include "layout.h"

struct vbq_matrix {
  int64_t N = 0, K = 0;
  int32_t G = 0;
  int32_t n_tiles = 0, n_steps = 0;
  int32_t max_tile_rows = 0;
  int64_t code_bytes = 0, meta_bytes = 0, total_bytes = 0, data_bytes = 0;
  int64_t groups_by_bits[4] = {0, 0, 0, 0};
  int device = 0;
  uint8_t* dev_base = nullptr;  // one allocation holding everything below
  const uint8_t* data = nullptr;
  const uint32_t* step_desc = nullptr;
  const uint32_t* step_off = nullptr;
  const uint32_t* tile_row0 = nullptr;
  const uint32_t* tile_step0 = nullptr;
  std::vector<uint32_t> h_tile_row0, h_tile_step0;
};

namespace vbq {

// Records the error detail for vbq_last_error() and returns the status.
vbq_status fail(vbq_status s, const std::string& detail);
vbq_status cuda_fail(cudaError_t e, const char* what);
void note_launches(int64_t n);

// Device-side check word (one int per device), set by kernels when a bounded wait runs out.
int* device_check_word();

struct GpuInfo {
  int device = -1;
  int sms = 0;
  int max_smem_optin = 0;
};
const GpuInfo& gpu_info();

}  // namespace vbq

#define VBQ_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return vbq::cuda_fail(_e, #expr); \
  } while (0)
