// Kernels and C-ABI entry points for vbq_dequant, vbq_gemv, vbq_gemm_smallbatch,
// the dense bf16 baseline, and the library's error and launch bookkeeping.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>

#include "gemv.cuh"
#include "internal.h"
#include "launch.h"

namespace vbq {

// ---------------------------------------------------------------- bookkeeping

static thread_local std::string g_last_error;
static std::atomic<int64_t> g_launches{0};

vbq_status fail(vbq_status s, const std::string& detail) {
  g_last_error = detail;
  return s;
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

MatView view_of(const vbq_matrix* m, float* y, int32_t y_ld, float* trace_y) {
  MatView v{};
  v.data = m->data;
  v.run_desc = m->run_desc;
  v.y = y;
  v.y_off = 0;
  v.y_ld = y_ld;
  v.trace_y = trace_y;
  return v;
}

PlanView plan_view(const DevicePlan& p) {
  PlanView v{};
  v.units = p.units;
  v.slices = p.slices;
  v.umax = p.umax;
  v.partial = p.partial;
  v.counters = p.counters;
  return v;
}

// ---------------------------------------------------------------- GEMV launch

// Kernel shapes: batch columns, warps per CTA, ring slots per warp.
template <int NB> struct GemvShape;
template <> struct GemvShape<1> { static constexpr int W = 16, NSLOT = 2; };
template <> struct GemvShape<2> { static constexpr int W = 16, NSLOT = 2; };
template <> struct GemvShape<4> { static constexpr int W = 8, NSLOT = 4; };

template <int NB>
struct GemvKernel {
  static constexpr int W = GemvShape<NB>::W, NSLOT = GemvShape<NB>::NSLOT;
  static constexpr int kThreads = W * 32;
  static constexpr int kSmem = GemvSmem<NB, W, NSLOT>::kBytes;
  static void prepare() {  // once per device
    static std::mutex mu;
    static std::map<int, bool> done;
    const GpuInfo& gi = gpu_info();
    std::lock_guard<std::mutex> lock(mu);
    if (done[gi.device]) return;
    cudaFuncSetAttribute(vbq_gemv_kernel<NB, W, NSLOT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    done[gi.device] = true;
  }
};

template <int NB>
cudaError_t launch_gemv_t(const GemvArgs& a, int n_ctas, cudaStream_t st, bool pdl) {
  using K = GemvKernel<NB>;
  K::prepare();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(n_ctas), 1, 1);
  cfg.blockDim = dim3(K::kThreads, 1, 1);
  cfg.dynamicSmemBytes = K::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  int na = 0;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, vbq_gemv_kernel<NB, K::W, K::NSLOT>, a);
}

cudaError_t launch_gemv(int nb, const GemvArgs& a, int n_ctas, cudaStream_t st, bool pdl) {
  if (n_ctas <= 0) return cudaSuccess;
  switch (nb) {
    case 1: return launch_gemv_t<1>(a, n_ctas, st, pdl);
    case 2: return launch_gemv_t<2>(a, n_ctas, st, pdl);
    case 4: return launch_gemv_t<4>(a, n_ctas, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

void warm_gemv(int nb) {
  switch (nb) {
    case 1: GemvKernel<1>::prepare(); break;
    case 2: GemvKernel<2>::prepare(); break;
    default: GemvKernel<4>::prepare(); break;
  }
}

// ---------------------------------------------------------------- dequant

// W[r][k] = s * (q - c_b) for every weight, exact in fp32. One CTA per tile;
// its warps take the tile's runs in turn.
__global__ void __launch_bounds__(256) vbq_dequant_kernel(const uint8_t* __restrict__ data,
                                                          const uint32_t* __restrict__ run_desc,
                                                          const uint32_t* __restrict__ run_off,
                                                          const uint32_t* __restrict__ tile_row0,
                                                          const uint32_t* __restrict__ tile_run0, int32_t K,
                                                          float* __restrict__ W) {
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint32_t r0 = tile_row0[t];
  for (uint32_t run = tile_run0[t] + warp; run < tile_run0[t + 1]; run += nw) {
    const uint32_t d = run_desc[run];
    const uint32_t cls = run_cls(d), n = run_n(d), g = run_g(d);
    const uint32_t eps = entries_per_step(cls);
    const uint8_t* rec = data + static_cast<uint64_t>(run_off[run]) * 16u;
    for (uint32_t k = 0; k * eps < n; ++k, rec += full_step_bytes(cls)) {
      const uint32_t e = min(eps, n - k * eps);
      const uint32_t j = static_cast<uint32_t>(lane);  // one entry per lane
      if (j >= e) continue;
      const uint32_t b = 1u << cls;
      const uint8_t* ent = rec + 8u * b * j;
      const float sc = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rec + rec_scale_off(cls, e) + 2 * j));
      const uint32_t row = rec[rec_row_off(cls, e) + j];
      const float c = static_cast<float>((1u << b) - 1u) * 0.5f;
      float* dst = W + static_cast<int64_t>(r0 + row) * K + static_cast<int64_t>(g) * GROUP;
      for (uint32_t m = 0; m < GROUP; ++m) {
        uint32_t q;
        if (b == 8) {
          q = ent[m];
        } else {
          q = 0;
          for (uint32_t p = 0; p < b; ++p) q |= ((ent[8 * p + (m >> 3)] >> (m & 7)) & 1u) << p;
        }
        dst[m] = __fmul_rn(sc, static_cast<float>(q) - c);
      }
    }
  }
}

// ---------------------------------------------------------------- dense bf16 baseline

// y = W x for a dense bf16 W [N][K]; one warp per row, x staged in shared memory.
__global__ void __launch_bounds__(256) vbq_dense_gemv_kernel(const uint16_t* __restrict__ W,
                                                             const uint16_t* __restrict__ x, float* __restrict__ y,
                                                             int32_t N, int32_t K) {
  extern __shared__ __align__(16) uint8_t xs_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(xs_raw);
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8)
    *reinterpret_cast<uint4*>(xs + k) = *reinterpret_cast<const uint4*>(x + k);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * nw + warp; r < N; r += static_cast<int64_t>(gridDim.x) * nw) {
    const uint16_t* wr = W + r * K;
    float acc0 = 0.f, acc1 = 0.f;
    int k = lane * 8;
#pragma unroll 1
    for (; k + 3 * 256 < K; k += 4 * 256) {
      uint4 wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) wv[u] = ldg_stream_v4(wr + k + u * 256);
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
  vbq_dequant_kernel<<<m->n_tiles, 256, 0, st>>>(m->data, m->run_desc, m->run_off, m->tile_row0, m->tile_run0,
                                                 static_cast<int32_t>(m->K), W_dev);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}

static vbq_status gemv_columns(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st) {
  if (m->N == 0) return VBQ_OK;
  if (m->K == 0) {
    VBQ_CUDA_TRY(cudaMemsetAsync(Y, 0, sizeof(float) * static_cast<size_t>(m->N) * B, st));
    return VBQ_OK;
  }
  int* err = device_check_word();
  if (!err) return fail(VBQ_ERR_CUDA, "device check word");
  int done = 0;
  while (done < B) {
    const int left = B - done;
    const int nb = left >= 4 ? 4 : left >= 2 ? 2 : 1;
    GemvArgs a{};
    a.it.seg[0] = view_of(m, Y + static_cast<int64_t>(done) * m->N, static_cast<int32_t>(m->N), nullptr);
    a.it.nseg = 1;
    a.it.plan = plan_view(m->plan);
    a.it.xs.mode = X_BF16;
    a.it.xs.K = static_cast<int32_t>(m->K);
    a.it.xs.x = X + static_cast<int64_t>(done) * m->K;
    a.it.xs.ldx = static_cast<int32_t>(m->K);
    a.it.ep = EP_STORE;
    a.err = err;
    const bool w8 = nb == 4;  // the 4-column kernel has 8 warps
    a.pieces = w8 ? m->plan.pieces8 : m->plan.pieces16;
    a.pstart = w8 ? m->plan.start8 : m->plan.start16;
    a.pbytes = w8 ? m->plan.bytes8 : m->plan.bytes16;
    VBQ_CUDA_TRY(launch_gemv(nb, a, m->plan.n_ctas, st, false));
    done += nb;
  }
  return VBQ_OK;
}

extern "C" vbq_status vbq_gemv(const vbq_matrix* m, const uint16_t* x_dev, float* y_dev, void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL matrix");
  if (m->N > 0 && !y_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL y");
  if (m->N > 0 && m->K > 0 && !x_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: NULL x");
  if (!aligned(x_dev, 4) || !aligned(y_dev, 4)) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemv: x and y must be 4-byte aligned");
  return gemv_columns(m, x_dev, 1, y_dev, static_cast<cudaStream_t>(stream));
}

extern "C" vbq_status vbq_gemm_smallbatch(const vbq_matrix* m, const uint16_t* X_dev, int32_t B, float* Y_dev,
                                          void* stream) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL matrix");
  if (B < 1 || B > 64) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: B must be in [1, 64]");
  if (m->N > 0 && !Y_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL Y");
  if (m->N > 0 && m->K > 0 && !X_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: NULL X");
  if (!aligned(X_dev, 4) || !aligned(Y_dev, 4))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_gemm_smallbatch: X and Y must be 4-byte aligned");
  // 16 or more columns form a dense contraction: the tensor-core dequant-MMA.
  if (B >= 16 && m->N > 0 && m->K > 0 && aligned(X_dev, 16) && tc_eligible(m))
    return launch_gemm_tc(m, X_dev, B, Y_dev, static_cast<cudaStream_t>(stream));
  return gemv_columns(m, X_dev, B, Y_dev, static_cast<cudaStream_t>(stream));
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
  vbq_dense_gemv_kernel<<<static_cast<unsigned>(grid), 256, smem, st>>>(W_dev, x_dev, y_dev, static_cast<int32_t>(N),
                                                                        static_cast<int32_t>(K));
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}
