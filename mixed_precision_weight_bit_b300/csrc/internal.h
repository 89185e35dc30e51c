// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/vbq.h"
#include "layout.h"
#include "plan.h"

// Device data of a plan for one batch-1 GEMV over one matrix.
struct GemvPlanDev {
  void* base = nullptr;         // one allocation for everything below
  const vbq::WarpPlan* warps = nullptr;
  const vbq::CtaPlan* ctas = nullptr;
  const uint32_t* arrivals = nullptr;  // per super-tile
  uint32_t* counters = nullptr;        // per super-tile, zero between calls
  unsigned long long* acc = nullptr;   // fixed-point row sums [n_super * 1024], zero between calls
  const uint64_t* pieces = nullptr;
  const uint32_t* pstart = nullptr;
  const uint32_t* pbytes = nullptr;
  int32_t n_ctas = 0;
  int64_t bytes = 0;
};

struct vbq_matrix {
  int64_t N = 0, K = 0;
  int32_t G = 0;
  int32_t n_tiles = 0;             // 256-row tiles
  int32_t n_super = 0;             // 1024-row super-tiles
  int64_t n_runs = 0;
  int64_t n_steps = 0;
  int64_t code_bytes = 0, meta_bytes = 0, total_bytes = 0, data_bytes = 0;
  int64_t groups_by_bits[4] = {0, 0, 0, 0};
  int device = 0;
  uint8_t* dev_base = nullptr;     // the packed stream
  const uint8_t* data = nullptr;
  const uint64_t* st_byte0 = nullptr;  // device [n_super + 1]: first byte of each super-tile's runs
  std::vector<vbq::RunInfo> runs;  // host copy of the run list, for planning
  std::vector<uint32_t> block_run; // [n_super * G + 1]: first run of each (super-tile, group column)
  float max_row_l1 = 0.0f;         // max over rows of sum_k |w_rk|, rounded up
  uint16_t max_scale_bits = 0;     // largest |s_g| as fp16 magnitude bits
  float max_scale = 0.0f;          // the same as a float
  GemvPlanDev gemv;                // batch-1 GEMV plan and its accumulators
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

// Device allocation of the library's buffers. Under the test hook
// VBQ_DEBUG_ALLOC_CAP a request above the cap fails with
// cudaErrorMemoryAllocation without reaching the driver.
cudaError_t dev_alloc(void** p, size_t bytes);
void set_alloc_cap(int64_t bytes);

// The decode step's attention input: rounds q, k, v of a [q;k;v] item's float
// output to bf16, turns q (into q_rot) and k (into the cache at pos) by the
// rotary embedding, and stores v at pos (attention.cu).
vbq_status launch_attn_prep(const float* qkv, int64_t q_off, int64_t k_off, int64_t v_off, uint16_t* q_rot,
                            uint16_t* k_cache, uint16_t* v_cache, int32_t H, int32_t Hkv, int32_t d, int64_t stride,
                            int32_t pos, double theta, cudaStream_t st);

// Tensor-core dequant-MMA for 2..64 batch columns (gemm_tc.cu).
bool tc_eligible(const vbq_matrix* m);
vbq_status launch_gemm_tc(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st);
void tc_forget(const vbq_matrix* m);

}  // namespace vbq

#define VBQ_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t _e = (expr);                                 \
    if (_e != cudaSuccess) return vbq::cuda_fail(_e, #expr); \
  } while (0)
