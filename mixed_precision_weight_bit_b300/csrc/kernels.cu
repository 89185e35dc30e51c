// Kernels and C-ABI entry points for vbq_dequant, vbq_gemv, vbq_gemm_smallbatch,
// the dense bf16 baseline, and the library's error and launch bookkeeping.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>

#include "gemv.cuh"
#include "internal.h"
#include <cstring>
#include <vector>

namespace vbq {

// ---------------------------------------------------------------- bookkeeping

static thread_local std::string g_last_error;
static std::atomic<int64_t> g_launches{0};

vbq_status fail(vbq_status s, const std::string& detail) {
  g_last_error = detail;
  return s;
}

static std::atomic<int64_t> g_alloc_cap{0};

void set_alloc_cap(int64_t bytes) { g_alloc_cap.store(bytes); }

cudaError_t dev_alloc(void** p, size_t bytes) {
  const int64_t cap = g_alloc_cap.load();
  if (cap > 0 && bytes > static_cast<size_t>(cap)) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

vbq_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  if (e == cudaErrorMemoryAllocation) return VBQ_ERR_OOM;
  return VBQ_ERR_CUDA;
}

void note_launches(int64_t n) { g_launches.fetch_add(n); }

int* device_check_word() {
  static std::mutex mu;
  static std::map<int, int*> words;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = words.find(dev);
  if (it != words.end()) return it->second;
  int* p = nullptr;
  if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return nullptr;
  if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return nullptr;
  words[dev] = p;
  return p;
}

const GpuInfo& gpu_info() {
  static std::mutex mu;
  static std::map<int, GpuInfo> infos;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = infos.find(dev);
  if (it != infos.end()) return it->second;
  GpuInfo gi;
  gi.device = dev;
  cudaDeviceGetAttribute(&gi.sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&gi.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return infos.emplace(dev, gi).first->second;
}

// ---- the single-GEMV kernel --------------------------------------------------

struct Gemv1Args {
  const WarpPlan* warps;
  const CtaPlan* ctas;
  const uint32_t* arrivals;  // per super-tile
  uint32_t* counters;        // per super-tile
  unsigned long long* acc;   // [n_super * 1024] fixed-point sums, zero between calls
  const uint64_t* pieces;
  const uint32_t* pstart;
  const uint32_t* pbytes;
  const uint16_t* x;         // bf16 [K]
  float* y;                  // [N]
  int64_t N;
  int32_t K;
  int32_t ns;                // ring slots per warp
  float max_row_l1;
  int* err;
};

__global__ void __launch_bounds__(KW * 32, 1) vbq_gemv1_kernel(const __grid_constant__ Gemv1Args a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SmemLayout L = smem_layout(a.ns);
  WarpStream S;
  Worker K;
  worker_init(S, K, L, static_cast<uint32_t>(a.ns), a.pieces, a.pstart, a.pbytes, lane, warp);
  for (uint32_t i = threadIdx.x; i < SLOTS_MAX * SROWS; i += KW * 32) sts<int>(L.acc + 4 * i, 0);
  const CtaPlan cp = a.ctas[blockIdx.x];

  // The weights do not depend on the previous kernel: the copies above already
  // run. Wait for it before reading x or touching the accumulators.
  grid_dep_launch();
  grid_dep_wait();

  float* red = reinterpret_cast<float*>(vbq_smem + L.misc);
  const int F = fixed_exponent(a.max_row_l1, max_abs_bf16(a.x, a.K, red));
  // Stage this CTA's columns; each warp issues all its loads first.
  const uint32_t na = cp.a1 - cp.a0;
  const uint32_t ncols = na + (cp.b1 - cp.b0);
  {
    stage_columns(L, ncols, F, lane, warp, [&](uint32_t j, float* x0, float* x1) {
      const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
      const uint32_t v = ldg_nc_u32(a.x + static_cast<size_t>(g) * GROUP + 2 * lane);
      *x0 = bf16_lo(v);
      *x1 = bf16_hi(v);
    });
  }
  __syncthreads();

  if (cp.n_slots > 0) warp_item(L, a.warps + static_cast<size_t>(blockIdx.x) * KW + warp, nullptr, cp, S, K, lane);
  if (!S.ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    S.drain();
  }
  __syncthreads();
  if (cp.n_slots == 0) return;
  flush_slots(L, cp, a.acc);
  __threadfence();
  __syncthreads();
  // The last CTA to add into a super-tile converts its rows and clears them for the next call.
  uint32_t* fin = reinterpret_cast<uint32_t*>(vbq_smem + L.misc) + 16;
  if (threadIdx.x == 0) {
    uint32_t nf = 0;
    for (uint32_t s = 0; s < cp.n_slots; ++s) {
      const uint32_t t = cp.st_base + s;
      if (atomicAdd(a.counters + t, 1u) == a.arrivals[t] - 1u) fin[1 + nf++] = t;
    }
    fin[0] = nf;
  }
  __syncthreads();
  const uint32_t nf = fin[0];
  if (nf == 0) return;
  __threadfence();
  for (uint32_t f = 0; f < nf; ++f) {
    const uint32_t t = fin[1 + f];
    for (uint32_t r = threadIdx.x; r < SROWS; r += KW * 32) {
      const int64_t row = static_cast<int64_t>(t) * SROWS + r;
      unsigned long long* p = a.acc + row;
      const long long v = static_cast<long long>(__ldcg(p));
      if (row < a.N) a.y[row] = scalbnf(__ll2float_rn(v), -F);
      *p = 0ull;
    }
    if (threadIdx.x == 0) a.counters[t] = 0u;
  }
}


static_assert(smem_layout(kRingSlots).total <= 232448, "shared memory");

static void prepare_gemv1() {
  static std::mutex mu;
  static std::map<int, bool> done;
  const GpuInfo& gi = gpu_info();
  std::lock_guard<std::mutex> lock(mu);
  if (done[gi.device]) return;
  cudaFuncSetAttribute(vbq_gemv1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_layout(kRingSlots).total);
  done[gi.device] = true;
}

// One batch-1 GEMV launch over matrix m (K <= XCAP, N > 0, K > 0).
static cudaError_t launch_gemv1(const vbq_matrix* m, const uint16_t* x, float* y, cudaStream_t st, int* err) {
  prepare_gemv1();
  const GemvPlanDev& P = m->gemv;
  Gemv1Args a{};
  a.warps = P.warps;
  a.ctas = P.ctas;
  a.arrivals = P.arrivals;
  a.counters = P.counters;
  a.acc = P.acc;
  a.pieces = P.pieces;
  a.pstart = P.pstart;
  a.pbytes = P.pbytes;
  a.x = x;
  a.y = y;
  a.N = m->N;
  a.K = static_cast<int32_t>(m->K);
  a.ns = kRingSlots;
  a.max_row_l1 = m->max_row_l1;
  a.err = err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.n_ctas), 1, 1);
  cfg.blockDim = dim3(KW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem_layout(kRingSlots).total;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, vbq_gemv1_kernel, a);
}

// ---------------------------------------------------------------- dequant

// W[r][k] = s * (q - c_b) for every weight, exact in fp32. One CTA per
// super-tile walks its runs in stream order; its threads share each step.
__global__ void __launch_bounds__(256) vbq_dequant_kernel(const uint8_t* __restrict__ data,
                                                          const uint64_t* __restrict__ st_byte0, int32_t K,
                                                          float* __restrict__ W) {
  const int t = blockIdx.x;
  uint64_t o = st_byte0[t];
  const uint64_t end = st_byte0[t + 1];
  while (o < end) {
    const RunHeader h = *reinterpret_cast<const RunHeader*>(data + o);
    o += HEADER_BYTES;
    const uint32_t cls = h.cls, n = h.n, b = 1u << cls;
    const uint32_t eps = entries_per_step(cls);
    const float c = static_cast<float>((1u << b) - 1u) * 0.5f;
    for (uint32_t done = 0; done < n; done += eps) {
      const uint32_t e = min(eps, n - done);
      const uint8_t* rec = data + o;
      for (uint32_t i = threadIdx.x; i < e * GROUP; i += blockDim.x) {
        const uint32_t j = i / GROUP, m = i % GROUP;
        const uint32_t per_word = 32u / b, r = m % per_word;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + code_word_off(cls, e, j, m / per_word));
        const uint32_t q = (w >> (b == 1 ? r : code_bit(b, r))) & ((1u << b) - 1u);
        const float sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rec + rec_scale_off(cls, e) + 2 * j));
        const uint32_t row = h.row0 + entry_tile(h, done + j) * TILE + rec[rec_row_off(cls, e) + j];
        W[static_cast<int64_t>(row) * K + static_cast<int64_t>(h.g) * GROUP + m] = __fmul_rn(sc, static_cast<float>(q) - c);
      }
      o += rec_bytes(cls, e);
    }
  }
}

// ---------------------------------------------------------------- dense bf16 baseline

// y = W x for a dense bf16 W [N][K]; one warp per row, x staged in shared memory.
// Launched with programmatic dependent launch: a CTA first issues the loads of
// its first row's weights, which do not depend on earlier kernels, then waits
// for the preceding grid's memory before it reads x; the next launch may start
// as soon as every CTA of this one has started.
__global__ void __launch_bounds__(256) vbq_dense_gemv_kernel(const uint16_t* __restrict__ W,
                                                             const uint16_t* __restrict__ x, float* __restrict__ y,
                                                             int32_t N, int32_t K) {
  extern __shared__ __align__(16) uint8_t xs_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(xs_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  grid_dep_launch();
  int64_t r = static_cast<int64_t>(blockIdx.x) * nw + warp;
  uint4 pre[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int k = lane * 8 + u * 256;
    pre[u] = (r < N && k < K) ? ldg_stream_v4(W + r * K + k) : make_uint4(0u, 0u, 0u, 0u);
  }
  grid_dep_wait();
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8)
    *reinterpret_cast<uint4*>(xs + k) = *reinterpret_cast<const uint4*>(x + k);
  __syncthreads();
  bool first = true;
  for (; r < N; r += static_cast<int64_t>(gridDim.x) * nw) {
    const uint16_t* wr = W + r * K;
    float acc0 = 0.f, acc1 = 0.f;
    int k = lane * 8;
#pragma unroll 1
    for (; k + 3 * 256 < K; k += 4 * 256) {
      uint4 wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) wv[u] = first ? pre[u] : ldg_stream_v4(wr + k + u * 256);
      first = false;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + k + u * 256);
        const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc0 = fmaf(bf16_lo(ww[q]), bf16_lo(xx[q]), acc0);
          acc1 = fmaf(bf16_hi(ww[q]), bf16_hi(xx[q]), acc1);
        }
      }
    }
    first = false;
    for (; k < K; k += 256) {
      const uint4 wv = ldg_stream_v4(wr + k);
      const uint4 xv = *reinterpret_cast<const uint4*>(xs + k);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
      const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc0 = fmaf(bf16_lo(ww[q]), bf16_lo(xx[q]), acc0);
        acc1 = fmaf(bf16_hi(ww[q]), bf16_hi(xx[q]), acc1);
      }
    }
    float v = acc0 + acc1;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if (lane == 0) y[r] = v;
  }
}

}  // namespace vbq

using namespace vbq;

// ---------------------------------------------------------------- C ABI

extern "C" const char* vbq_status_str(vbq_status s) {
  switch (s) {
    case VBQ_OK: return "VBQ_OK";
    case VBQ_ERR_INVALID_ARG: return "VBQ_ERR_INVALID_ARG";
    case VBQ_ERR_SHAPE: return "VBQ_ERR_SHAPE";
    case VBQ_ERR_CODE_RANGE: return "VBQ_ERR_CODE_RANGE";
    case VBQ_ERR_BITS: return "VBQ_ERR_BITS";
    case VBQ_ERR_CUDA: return "VBQ_ERR_CUDA";
    case VBQ_ERR_OOM: return "VBQ_ERR_OOM";
    case VBQ_ERR_DEVICE_CHECK: return "VBQ_ERR_DEVICE_CHECK";
    case VBQ_ERR_UNSUPPORTED: return "VBQ_ERR_UNSUPPORTED";
  }
  return "VBQ_ERR_UNKNOWN";
}

extern "C" const char* vbq_last_error(void) { return g_last_error.c_str(); }

extern "C" int64_t vbq_launch_count(int32_t reset) {
  return reset ? g_launches.exchange(0) : g_launches.load();
}

extern "C" vbq_status vbq_device_check(int32_t* code) {
  int* w = device_check_word();
  if (!w) return fail(VBQ_ERR_CUDA, "vbq_device_check: no device word");
  VBQ_CUDA_TRY(cudaDeviceSynchronize());
  int v = 0;
  VBQ_CUDA_TRY(cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost));
  VBQ_CUDA_TRY(cudaMemset(w, 0, sizeof(int)));
  if (code) *code = v;
  return v ? fail(VBQ_ERR_DEVICE_CHECK, "a kernel's bounded wait ran out (code " + std::to_string(v) + ")") : VBQ_OK;
}

static inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

extern "C" vbq_status vbq_dequant(const vbq_matrix* m, float* W_dev, void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_dequant: NULL matrix");
  if (m->N * m->K == 0) return VBQ_OK;
  if (!W_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_dequant: NULL output");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  note_launches(1);
  vbq_dequant_kernel<<<m->n_super, 256, 0, st>>>(m->data, m->st_byte0, static_cast<int32_t>(m->K), W_dev);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}

// Batch columns one at a time through the batch-1 kernel (each call streams the
// matrix once); from VBQ_TC_MIN_BATCH columns on, the tensor-core path.
#ifndef VBQ_TC_MIN_BATCH
#define VBQ_TC_MIN_BATCH 4
#endif
static constexpr int32_t kTcMinBatch = VBQ_TC_MIN_BATCH;

static vbq_status gemv_columns(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st) {
  if (m->N == 0) return VBQ_OK;
  if (m->K == 0) {
    VBQ_CUDA_TRY(cudaMemsetAsync(Y, 0, sizeof(float) * static_cast<size_t>(m->N) * B, st));
    return VBQ_OK;
  }
  if (m->K > XCAP) return fail(VBQ_ERR_UNSUPPORTED, "K above 16384 on the batch-1 path");
  int* err = device_check_word();
  if (!err) return fail(VBQ_ERR_CUDA, "device check word");
  for (int j = 0; j < B; ++j)
    VBQ_CUDA_TRY(launch_gemv1(m, X + static_cast<int64_t>(j) * m->K, Y + static_cast<int64_t>(j) * m->N, st, err));
  return VBQ_OK;
}

extern "C" vbq_status vbq_gemv(const vbq_matrix* m, const uint16_t* x_dev, float* y_dev, void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL matrix");
  if (m->N > 0 && !y_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL y");
  if (m->N > 0 && m->K > 0 && !x_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL x");
  if (!aligned(x_dev, 4) || !aligned(y_dev, 4)) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: x and y must be 4-byte aligned");
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: matrix is on another device");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (m->K > XCAP && m->N > 0) {
    if (!tc_eligible(m)) return fail(VBQ_ERR_UNSUPPORTED, "vbq_gemv: K above 16384 needs the tensor-core path");
    return launch_gemm_tc(m, x_dev, 1, y_dev, st);
  }
  return gemv_columns(m, x_dev, 1, y_dev, st);
}

extern "C" vbq_status vbq_gemm_smallbatch(const vbq_matrix* m, const uint16_t* X_dev, int32_t B, float* Y_dev,
                                          void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL matrix");
  if (B < 1 || B > 64) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: B must be in [1, 64]");
  if (m->N > 0 && !Y_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL Y");
  if (m->N > 0 && m->K > 0 && !X_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL X");
  if (!aligned(X_dev, 4) || !aligned(Y_dev, 4))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: X and Y must be 4-byte aligned");
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: matrix is on another device");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Two or more columns form a dense contraction: the tensor-core dequant-MMA decodes each code once.
  // Batches of 4 and more take the tensor cores: their cost hardly depends on B, and on 14336x4096 at
  // the config-0 allocation it is below four batch-1 GEMVs (measured crossover between 3 and 4).
  if (B >= kTcMinBatch && m->N > 0 && m->K > 0 && tc_eligible(m)) return launch_gemm_tc(m, X_dev, B, Y_dev, st);
  if (B == 1 && m->K > XCAP && m->N > 0 && tc_eligible(m)) return launch_gemm_tc(m, X_dev, 1, Y_dev, st);
  return gemv_columns(m, X_dev, B, Y_dev, st);
}

// Many dense GEMVs, one persistent launch: global row r (rows of all jobs in
// job order) goes to warp r mod (warps of the grid); x is read through L1,
// where the rows of one job that a CTA's warps take in turn find it.
struct DenseManyArgs {
  const uint16_t* W[VBQ_DENSE_MAX_JOBS];
  const uint16_t* x[VBQ_DENSE_MAX_JOBS];
  float* y[VBQ_DENSE_MAX_JOBS];
  int32_t K[VBQ_DENSE_MAX_JOBS];
  int64_t row0[VBQ_DENSE_MAX_JOBS + 1];  // first global row of each job; row0[n] = all rows
  int32_t n;
};
static_assert(sizeof(DenseManyArgs) < 32000, "kernel parameter space");

constexpr int kDenseWarps = 8;  // per CTA
constexpr int kDenseUnroll = 8;  // 16-byte loads in flight per lane

__global__ void __launch_bounds__(kDenseWarps * 32, 3) vbq_dense_many_kernel(const __grid_constant__ DenseManyArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kDenseWarps, total = a.row0[a.n];
  grid_dep_wait();
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kDenseWarps + warp; r < total; r += stride) {
    int lo = 0, hi = a.n - 1;  // the job: the last with row0 <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.row0[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int K = a.K[lo];
    const uint16_t* wr = a.W[lo] + (r - a.row0[lo]) * K;
    const uint16_t* x = a.x[lo];
    float acc0 = 0.f, acc1 = 0.f;
    int k = lane * 8;
    for (; k + (kDenseUnroll - 1) * 256 < K; k += kDenseUnroll * 256) {
      uint4 wv[kDenseUnroll], xv[kDenseUnroll];
#pragma unroll
      for (int u = 0; u < kDenseUnroll; ++u) wv[u] = ldg_stream_v4(wr + k + u * 256);
#pragma unroll
      for (int u = 0; u < kDenseUnroll; ++u) xv[u] = __ldg(reinterpret_cast<const uint4*>(x + k + u * 256));
#pragma unroll
      for (int u = 0; u < kDenseUnroll; ++u) {
        const uint32_t ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        const uint32_t xx[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc0 = fmaf(bf16_lo(ww[q]), bf16_lo(xx[q]), acc0);
          acc1 = fmaf(bf16_hi(ww[q]), bf16_hi(xx[q]), acc1);
        }
      }
    }
    for (; k < K; k += 256) {
      const uint4 wv = ldg_stream_v4(wr + k);
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + k));
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
      const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc0 = fmaf(bf16_lo(ww[q]), bf16_lo(xx[q]), acc0);
        acc1 = fmaf(bf16_hi(ww[q]), bf16_hi(xx[q]), acc1);
      }
    }
    float v = acc0 + acc1;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    if (lane == 0) a.y[lo][r - a.row0[lo]] = v;
  }
}

extern "C" vbq_status vbq_gemm(const vbq_matrix* m, const uint16_t* X_dev, int64_t B, float* Y_dev, void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm: NULL matrix");
  if (B < 1 || B > (int64_t(1) << 24)) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm: B must be in [1, 2^24]");
  // Blocks of 64 columns, each one vbq_gemm_smallbatch call (the tensor cores from 4 columns on).
  for (int64_t b0 = 0; b0 < B; b0 += 64) {
    const int32_t nb = static_cast<int32_t>(B - b0 < 64 ? B - b0 : 64);
    const vbq_status s = vbq_gemm_smallbatch(m, X_dev ? X_dev + b0 * m->K : nullptr, nb,
                                             Y_dev ? Y_dev + b0 * m->N : nullptr, stream);
    if (s != VBQ_OK) return s;
  }
  return VBQ_OK;
}

extern "C" vbq_status vbq_dense_gemv_bf16_many(const vbq_dense_job* jobs, int32_t n_jobs, void* stream) {
  if (n_jobs < 0 || n_jobs > VBQ_DENSE_MAX_JOBS)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16_many: n_jobs out of range");
  if (n_jobs > 0 && !jobs) return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16_many: NULL jobs");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int32_t j = 0; j < n_jobs; ++j) {
    const vbq_dense_job& d = jobs[j];
    if (d.N < 0 || d.K < 0 || d.K % 8 || d.N >= (int64_t(1) << 31) || d.K >= (int64_t(1) << 31))
      return fail(VBQ_ERR_SHAPE, "vbq_dense_gemv_bf16_many: need K % 8 == 0 and N, K < 2^31");
    if (d.N > 0 && !d.y) return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16_many: NULL y");
    if (d.N > 0 && d.K > 0 && (!d.W || !d.x || !aligned(d.W, 16) || !aligned(d.x, 16)))
      return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16_many: W and x must be 16-byte aligned device buffers");
  }
  DenseManyArgs a{};
  int64_t rows = 0;
  for (int32_t j = 0; j < n_jobs; ++j) {
    const vbq_dense_job& d = jobs[j];
    if (d.N == 0) continue;
    if (d.K == 0) {
      VBQ_CUDA_TRY(cudaMemsetAsync(d.y, 0, sizeof(float) * d.N, st));
      continue;
    }
    a.W[a.n] = d.W;
    a.x[a.n] = d.x;
    a.y[a.n] = d.y;
    a.K[a.n] = static_cast<int32_t>(d.K);
    a.row0[a.n] = rows;
    rows += d.N;
    ++a.n;
  }
  a.row0[a.n] = rows;
  if (a.n == 0) return VBQ_OK;
  int64_t grid = (rows + kDenseWarps - 1) / kDenseWarps;
  const int64_t cap = static_cast<int64_t>(gpu_info().sms) * 3;
  if (grid > cap) grid = cap;
  note_launches(1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kDenseWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_dense_many_kernel, a));
  return VBQ_OK;
}

extern "C" vbq_status vbq_dense_gemv_bf16(const uint16_t* W_dev, const uint16_t* x_dev, float* y_dev, int64_t N,
                                          int64_t K, void* stream) {
  if (N < 0 || K < 0 || K % 8 || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return fail(VBQ_ERR_SHAPE, "vbq_dense_gemv_bf16: need K % 8 == 0 and N, K < 2^31");
  if (N == 0) return VBQ_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!y_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16: NULL y");
  if (K == 0) {
    VBQ_CUDA_TRY(cudaMemsetAsync(y_dev, 0, sizeof(float) * N, st));
    return VBQ_OK;
  }
  if (!W_dev || !x_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16: NULL input");
  if (!aligned(W_dev, 16) || !aligned(x_dev, 16))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_dense_gemv_bf16: W and x must be 16-byte aligned");
  const size_t smem = static_cast<size_t>(K) * 2;
  if (smem > static_cast<size_t>(gpu_info().max_smem_optin))
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_dense_gemv_bf16: K too large for shared-memory staging");
  static std::once_flag once;
  std::call_once(once, [&]() {
    cudaFuncSetAttribute(vbq_dense_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         gpu_info().max_smem_optin);
  });
  const int64_t warps = (N + 0);
  int64_t grid = (warps + 7) / 8;
  const int64_t cap = static_cast<int64_t>(gpu_info().sms) * 16;
  if (grid > cap) grid = cap;
  note_launches(1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_dense_gemv_kernel, W_dev, x_dev, y_dev, static_cast<int32_t>(N),
                                  static_cast<int32_t>(K)));
  return VBQ_OK;
}
