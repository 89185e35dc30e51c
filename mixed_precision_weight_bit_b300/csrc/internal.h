// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/vbq.h"
#include "layout.h"
#include "plan.h"

struct vbq_matrix {
  int64_t N = 0, K = 0;
  int32_t G = 0;
  int32_t n_tiles = 0, n_runs = 0;
  int64_t n_steps = 0;
  int64_t code_bytes = 0, meta_bytes = 0, total_bytes = 0, data_bytes = 0;
  int64_t groups_by_bits[4] = {0, 0, 0, 0};
  int device = 0;
  uint8_t* dev_base = nullptr;  // one allocation: records and side tables
  const uint8_t* data = nullptr;
  const uint32_t* run_desc = nullptr;
  const uint32_t* run_off = nullptr;
  const uint32_t* tile_row0 = nullptr;
  const uint32_t* tile_run0 = nullptr;
  std::vector<uint32_t> h_run_desc, h_run_off, h_tile_row0, h_tile_run0;  // host copies, for planning
  vbq::DevicePlan plan;  // plan of a GEMV over this matrix alone
  float tc_max_scale = 0.0f;  // largest |s_g|: the tensor-core path needs s * 127.5 inside fp16
  int64_t max_col_bytes = 0;  // largest (tile, group column) record span
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

// Widest batch a single GEMV launch covers (partial storage is sized for it).
constexpr int MAX_NB = 4;

// Tensor-core dequant-MMA for 16..64 batch columns (gemm_tc.cu).
bool tc_eligible(const vbq_matrix* m);
vbq_status launch_gemm_tc(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st);
void tc_forget(const vbq_matrix* m);

inline SegTables seg_tables(const vbq_matrix* m) {
  SegTables t;
  t.run_desc = m->h_run_desc.data();
  t.run_off = m->h_run_off.data();
  t.tile_row0 = m->h_tile_row0.data();
  t.tile_run0 = m->h_tile_run0.data();
  t.n_tiles = m->n_tiles;
  t.n_runs = m->n_runs;
  return t;
}

}  // namespace vbq

#define VBQ_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return vbq::cuda_fail(_e, #expr); \
  } while (0)
