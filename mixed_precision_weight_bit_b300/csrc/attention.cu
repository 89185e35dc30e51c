// Decode attention over a bf16 KV cache, for one new token: rotary position
// embedding of q and k with the append of (k, v) to the cache, then grouped-
// query attention of every q head over positions 0 .. T-1.
//
// The source pages only say that the method speeds up token-by-token
// (autoregressive) decode; attention is the other half of a decode step
// beside the projections. What is computed here is the standard definition:
//  * rotary embedding, the rotate-half pairing: for i < d/2 the pair
//    (x_i, x_{i+d/2}) turns by the angle pos * theta^(-2i/d);
//  * scaled dot-product attention, scores q_h . k_j / sqrt(d), a softmax over
//    j < T, and the p-weighted sum of the v_j; query head h reads kv head
//    h / (H / H_kv).
//
// Work split (split-KV decoding): each kv head's positions are cut into at
// most kAttnMaxParts contiguous spans, one CTA per (span, kv head), about three
// CTAs per SM in all (what their shared memory allows; more CTAs per SM, with
// smaller or more buffers, measured slower). A CTA streams its span through
// kAttnBufs shared-memory buffers of kAttnSub positions (bulk copies of K and
// V, the next sub-chunk landing while one is used) and keeps, for each head of
// the group, a running softmax: the max score so far, the sum of exp, and the
// p-weighted sum of v, rescaled when the max grows. The last CTA of a kv head
// to finish (an atomic counter) merges the spans in span order, so results do
// not depend on timing. The cache is read from HBM once; what paces a CTA is
// its per-sub-chunk work (scores, softmax, weighted sums) between barriers.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace vbq {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnSub = 64;            // positions per sub-chunk (one buffer)
constexpr int kAttnBufs = 2;            // buffers: the next sub-chunk lands while one is used
constexpr int kAttnMaxGroup = 8;        // query heads per kv head
constexpr int kAttnMaxT = 65536;        // positions
constexpr int kAttnMaxParts = 64;       // spans per kv head
constexpr int kErrAttnCopyTimeout = 5;  // device check code: a sub-chunk copy never landed

struct AttnArgs {
  const uint16_t* q;        // bf16 [H][d]
  const uint16_t* k;        // bf16 [H_kv][stride][d]
  const uint16_t* v;
  float* out;               // [H][d]
  float* part;              // per (kv head, span, group head): max, sum, -, -, then d weighted sums
  uint32_t* counters;       // per kv head, zero between calls
  int64_t stride;           // positions allocated per kv head
  int32_t T, G, nparts, span;  // span: positions per CTA (a multiple of kAttnSub)
  float scale;              // 1/sqrt(d)
  int* err;
};

template <int HD>
struct AttnSmem {
  static constexpr int kBuf = kAttnSub * HD * 2 * 2;            // one buffer: K then V, bf16 [kAttnSub][HD] each
  static constexpr int kS = kAttnBufs * kBuf;                   // float [G][kAttnSub]: scores, then exp
  static constexpr int kW = 0;                                  // the merge's float [G][kAttnMaxParts], over buffer 0
  static_assert(kAttnMaxGroup * kAttnMaxParts * 4 <= kBuf, "merge weights fit over a buffer");
  static constexpr int kRed = kS + kAttnMaxGroup * kAttnSub * 4;  // float2 [G][HD/2]: the replicas' sum
  static constexpr int kStat = kRed + kAttnMaxGroup * HD * 4;   // float [G][4]: max, sum, rescale, -
  static constexpr int kBar = kStat + kAttnMaxGroup * 4 * 4;    // an mbarrier per buffer
  static constexpr int kFlag = kBar + 8 * kAttnBufs;
  static constexpr int kBytes = kFlag + 16;
};
constexpr int part_stride(int hd) { return hd + 4; }

extern __shared__ __align__(128) uint8_t attn_smem[];

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 3) vbq_attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  using L = AttnSmem<HD>;
  constexpr int NQ = HD / 64;             // 16-byte pieces of a row per lane in the score phase
  constexpr int NU = HD / 2;              // output threads per replica: one pair of dims each
  constexpr int R = kAttnThreads / NU;    // replicas: they split a sub-chunk's positions
  static_assert(kAttnThreads % NU == 0, "whole replicas");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, sub = lane >> 3, li = lane & 7;
  const int c = blockIdx.x, g = blockIdx.y, G = a.G;
  const int p0 = c * a.span, p1 = min(a.T, p0 + a.span);
  const int nsub = (p1 - p0 + kAttnSub - 1) / kAttnSub;
  const uint32_t sb = smem_u32(attn_smem);
  float* S = reinterpret_cast<float*>(attn_smem + L::kS);
  float2* red = reinterpret_cast<float2*>(attn_smem + L::kRed);
  float* stat = reinterpret_cast<float*>(attn_smem + L::kStat);
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(attn_smem + L::kFlag);
  const uint32_t bar0 = sb + L::kBar;

  // Sub-chunk t of the span into buffer t % kAttnBufs (thread 0).
  auto issue = [&](int t) {
    const int j0 = p0 + t * kAttnSub, np = min(kAttnSub, p1 - j0);
    const int b = t % kAttnBufs;
    const uint32_t bytes = static_cast<uint32_t>(np) * HD * 2u, buf = sb + b * L::kBuf;
    const size_t row = (static_cast<size_t>(g) * a.stride + j0) * HD;
    mbar_arrive_expect_tx(bar0 + 8 * b, 2u * bytes);
    bulk_g2s_plain(buf, a.k + row, bytes, bar0 + 8 * b);
    bulk_g2s_plain(buf + kAttnSub * HD * 2, a.v + row, bytes, bar0 + 8 * b);
  };
  grid_dep_wait();
  if (tid == 0) {
    for (int b = 0; b < kAttnBufs; ++b) mbar_init(bar0 + 8 * b, 1);
    fence_mbarrier_init();
    for (int t = 0; t < kAttnBufs - 1 && t < nsub; ++t) issue(t);
  }
  if (tid < kAttnMaxGroup) {
    stat[4 * tid] = -INFINITY;
    stat[4 * tid + 1] = 0.0f;
  }
  // Score work: warp w takes head hw = w / wph of the group (wph = 8 / G warps
  // per head) and positions wi * 4 + sub, + 4 wph, ... (wi = w % wph), 8 lanes
  // per position. Its head's query stays in registers, as fp32: lane li holds
  // dims [8 li, 8 li + 8) and, for d = 128, [64 + 8 li, ...).
  const int wph = (kAttnThreads / 32) / G, hw = warp / wph, wi = warp - hw * wph;
  const bool scorer = hw < G;
  float qv[NQ * 8];
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
    const uint4 w = scorer ? *reinterpret_cast<const uint4*>(a.q + (g * G + hw) * HD + 64 * n + 8 * li)
                           : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qv[8 * n + 2 * e] = __uint_as_float(ww[e] << 16);
      qv[8 * n + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    }
  }
  // Output: thread (r, dp) keeps, for every head of the group, the running
  // p-weighted sum of v's dims 2 dp, 2 dp + 1 over positions r, r + R, ...
  const int dp = tid % NU, rr = tid / NU;
  float2 acc[kAttnMaxGroup];
#pragma unroll
  for (int h = 0; h < kAttnMaxGroup; ++h) acc[h] = make_float2(0.0f, 0.0f);
  __syncthreads();  // the barriers and the running statistics

  bool ok = true;
  for (int t = 0; t < nsub && ok; ++t) {
    if (tid == 0 && t + kAttnBufs - 1 < nsub) {
      fence_proxy_async_smem();  // every thread's reads of that buffer (sub-chunk t - 1) ended before the last barrier
      issue(t + kAttnBufs - 1);
    }
    ok = mbar_wait(bar0 + 8 * (t % kAttnBufs), (t / kAttnBufs) & 1);
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    const uint8_t* Kb = attn_smem + (t % kAttnBufs) * L::kBuf;
    const uint32_t* V32 = reinterpret_cast<const uint32_t*>(Kb + kAttnSub * HD * 2);
    const int np = min(kAttnSub, p1 - (p0 + t * kAttnSub));
    // Scores: 8 lanes per position; each 16-byte shared load of a row is
    // conflict-free; two FMA chains, then a 3-step butterfly over the 8 lanes.
    if (scorer) {
      for (int base = wi * 4; base < np; base += 4 * wph) {
        const int j = base + sub;
        const bool valid = j < np;
        const uint8_t* row = Kb + (valid ? j : 0) * HD * 2;
        float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + 128 * n + 16 * li);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            d0 = fmaf(qv[8 * n + 2 * e], __uint_as_float(ww[e] << 16), d0);
            d1 = fmaf(qv[8 * n + 2 * e + 1], __uint_as_float(ww[e] & 0xFFFF0000u), d1);
          }
        }
        float d = d0 + d1;
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if (li == 0 && valid) S[hw * kAttnSub + j] = d * a.scale;
      }
    }
    __syncthreads();
    // Running softmax: warp h updates head h's max, rescale and sum.
    if (warp < G) {
      float m = -INFINITY;
      for (int j = lane; j < np; j += 32) m = fmaxf(m, S[warp * kAttnSub + j]);
      m = fmaxf(warp_max(m), stat[4 * warp]);
      float l = 0.0f;
      for (int j = lane; j < np; j += 32) {
        const float p = expf(S[warp * kAttnSub + j] - m);
        S[warp * kAttnSub + j] = p;
        l += p;
      }
      l = warp_sum(l);
      __syncwarp();
      if (lane == 0) {
        const float alpha = expf(stat[4 * warp] - m);  // 0 on the first sub-chunk (max -inf)
        stat[4 * warp] = m;
        stat[4 * warp + 1] = fmaf(stat[4 * warp + 1], alpha, l);
        stat[4 * warp + 2] = alpha;
      }
    }
    __syncthreads();
    // p-weighted sums of v, the old ones rescaled; v converted once for all heads.
    {
      float al[kAttnMaxGroup];
#pragma unroll
      for (int h = 0; h < kAttnMaxGroup; ++h) al[h] = h < G ? stat[4 * h + 2] : 0.0f;
#pragma unroll
      for (int h = 0; h < kAttnMaxGroup; ++h) {
        acc[h].x *= al[h];
        acc[h].y *= al[h];
      }
      for (int j = rr; j < np; j += R) {
        const uint32_t vv = V32[j * (HD / 2) + dp];
        const float vx = __uint_as_float(vv << 16), vy = __uint_as_float(vv & 0xFFFF0000u);
#pragma unroll
        for (int h = 0; h < kAttnMaxGroup; ++h) {
          if (h >= G) break;
          const float p = S[h * kAttnSub + j];
          acc[h].x = fmaf(p, vx, acc[h].x);
          acc[h].y = fmaf(p, vy, acc[h].y);
        }
      }
    }
    __syncthreads();  // buffer t % kAttnBufs is free for sub-chunk t + kAttnBufs; S and the rescales for the next step
  }
  if (!ok) {
    if (tid == 0) atomicExch(a.err, kErrAttnCopyTimeout);
    return;  // the barrier wait gave up everywhere at once (__syncthreads_and)
  }
  // The replicas' sums, added in replica order into red[h][dp].
  for (int r = 0; r < R; ++r) {
    if (rr == r)
#pragma unroll
      for (int h = 0; h < kAttnMaxGroup; ++h) {
        if (h >= G) break;
        float2 o = acc[h];
        if (r > 0) {
          const float2 t2 = red[h * NU + dp];
          o = make_float2(t2.x + o.x, t2.y + o.y);
        }
        red[h * NU + dp] = o;
      }
    __syncthreads();
  }
  // This CTA's span result for (h, pair dp).
  float* part = a.part + (static_cast<size_t>(g) * a.nparts + c) * kAttnMaxGroup * part_stride(HD);
  const bool single = a.nparts == 1;
  for (int u = tid; u < G * NU; u += kAttnThreads) {
    const int h = u / NU, d2 = u - h * NU;
    const float2 o = red[u];
    if (single) {
      const float inv = 1.0f / stat[4 * h + 1];
      a.out[(g * G + h) * HD + 2 * d2] = o.x * inv;
      a.out[(g * G + h) * HD + 2 * d2 + 1] = o.y * inv;
    } else {
      float* ph = part + h * part_stride(HD);
      ph[4 + 2 * d2] = o.x;
      ph[4 + 2 * d2 + 1] = o.y;
      if (d2 == 0) {
        ph[0] = stat[4 * h];
        ph[1] = stat[4 * h + 1];
      }
    }
  }
  if (single) return;

  // The last CTA of kv head g merges the spans in span order.
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = atomicAdd(a.counters + g, 1u) + 1u == static_cast<uint32_t>(a.nparts) ? 1u : 0u;
  __syncthreads();
  if (*flag == 0u) return;
  __threadfence();
  const float* pg = a.part + static_cast<size_t>(g) * a.nparts * kAttnMaxGroup * part_stride(HD);
  float* Wm = reinterpret_cast<float*>(attn_smem + L::kW);  // over buffer 0, no longer read
  // Per head: M = max over spans, the span weights exp(m_c - M) (in Wm), and L.
  if (warp < G) {
    float M = -INFINITY;
    for (int k = lane; k < a.nparts; k += 32) M = fmaxf(M, __ldcg(pg + (k * kAttnMaxGroup + warp) * part_stride(HD)));
    M = warp_max(M);
    float Ls = 0.0f;  // lane l sums spans l, l + 32, ...; then a fixed butterfly
    for (int k = lane; k < a.nparts; k += 32) {
      const float* pk = pg + (k * kAttnMaxGroup + warp) * part_stride(HD);
      const float w = expf(__ldcg(pk) - M);
      Wm[warp * kAttnMaxParts + k] = w;
      Ls = fmaf(w, __ldcg(pk + 1), Ls);
    }
    Ls = warp_sum(Ls);
    if (lane == 0) stat[4 * warp + 1] = Ls;
  }
  __syncthreads();
  for (int u = tid; u < G * HD; u += kAttnThreads) {
    const int h = u / HD, d = u - h * HD;
    float o = 0.0f;
#pragma unroll 8
    for (int k = 0; k < a.nparts; ++k)
      o = fmaf(Wm[h * kAttnMaxParts + k], __ldcg(pg + (k * kAttnMaxGroup + h) * part_stride(HD) + 4 + d), o);
    a.out[(g * G + h) * HD + d] = o / stat[4 * h + 1];
  }
  if (tid == 0) a.counters[g] = 0u;
}

// Rotary embedding at position pos (in fp64, rounded to fp32, then to bf16):
// block b < H turns q head b in place; block H + g turns k_new[g] into the
// cache at pos and copies v_new[g] there. Thread i takes the pair (i, i + d/2).
__global__ void vbq_rope_append_kernel(uint16_t* __restrict__ q, const uint16_t* __restrict__ k_new,
                                       const uint16_t* __restrict__ v_new, uint16_t* __restrict__ k_cache,
                                       uint16_t* __restrict__ v_cache, int32_t H, int32_t d, int64_t stride,
                                       int32_t pos, double theta) {
  const int b = blockIdx.x, i = threadIdx.x, half = d / 2;
  if (i >= half) return;
  const double inv_freq = pow(theta, -2.0 * i / d);
  double s, c;
  sincos(static_cast<double>(pos) * inv_freq, &s, &c);
  grid_dep_wait();  // the angles above need nothing from the kernel before; q, k and v do
  auto turn = [&](const uint16_t* src, uint16_t* dst) {
    const double x0 = __uint_as_float(static_cast<uint32_t>(src[i]) << 16);
    const double x1 = __uint_as_float(static_cast<uint32_t>(src[i + half]) << 16);
    const float y0 = __double2float_rn(x0 * c - x1 * s);
    const float y1 = __double2float_rn(x0 * s + x1 * c);
    dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(y0));
    dst[i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(y1));
  };
  if (b < H) {
    turn(q + static_cast<size_t>(b) * d, q + static_cast<size_t>(b) * d);
  } else {
    const int g = b - H;
    const size_t at = (static_cast<size_t>(g) * stride + pos) * d;
    turn(k_new + static_cast<size_t>(g) * d, k_cache + at);
    v_cache[at + i] = v_new[static_cast<size_t>(g) * d + i];
    v_cache[at + i + half] = v_new[static_cast<size_t>(g) * d + i + half];
  }
}

// The decode step's attention input (vbq_decode_step_at): q, k and v from a
// [q;k;v] item's float output (rows q_off.., k_off.., v_off..), each rounded to
// bf16 (nearest even) as the cache stores them; then block b < H turns q head
// b into q_rot, and block H + g turns k head g into the cache at pos and
// stores v head g there (the rotation of vbq_rope_append).
__global__ void vbq_attn_prep_kernel(const float* __restrict__ qkv, int64_t q_off, int64_t k_off, int64_t v_off,
                                     uint16_t* __restrict__ q_rot, uint16_t* __restrict__ k_cache,
                                     uint16_t* __restrict__ v_cache, int32_t H, int32_t d, int64_t stride, int32_t pos,
                                     double theta) {
  const int b = blockIdx.x, i = threadIdx.x, half = d / 2;
  if (i >= half) return;
  const double inv_freq = pow(theta, -2.0 * i / d);
  double s, c;
  sincos(static_cast<double>(pos) * inv_freq, &s, &c);
  grid_dep_wait();  // the angles above need nothing from the kernel before; q, k and v do
  auto bf = [](float v) { return __float2bfloat16_rn(v); };
  auto turn = [&](const float* src, uint16_t* dst) {
    const double x0 = __bfloat162float(bf(src[i])), x1 = __bfloat162float(bf(src[i + half]));
    dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__double2float_rn(x0 * c - x1 * s)));
    dst[i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(__double2float_rn(x0 * s + x1 * c)));
  };
  if (b < H) {
    turn(qkv + q_off + static_cast<int64_t>(b) * d, q_rot + static_cast<size_t>(b) * d);
  } else {
    const int g = b - H;
    const size_t at = (static_cast<size_t>(g) * stride + pos) * d;
    turn(qkv + k_off + static_cast<int64_t>(g) * d, k_cache + at);
    v_cache[at + i] = __bfloat16_as_ushort(bf(qkv[v_off + static_cast<int64_t>(g) * d + i]));
    v_cache[at + i + half] = __bfloat16_as_ushort(bf(qkv[v_off + static_cast<int64_t>(g) * d + i + half]));
  }
}

// Per-device scratch of the attention merge: partial results and counters.
struct AttnScratch {
  float* part = nullptr;
  uint32_t* counters = nullptr;
  size_t part_floats = 0;
  int32_t n_counters = 0;
};
std::mutex g_attn_mu;
std::map<int, AttnScratch> g_attn;

vbq_status attn_scratch(int dev, size_t part_floats, int32_t n_counters, AttnScratch** out) {
  std::lock_guard<std::mutex> lock(g_attn_mu);
  AttnScratch& s = g_attn[dev];
  if (s.part_floats < part_floats) {
    if (s.part) {
      VBQ_CUDA_TRY(cudaDeviceSynchronize());
      cudaFree(s.part);
      s.part = nullptr;
      s.part_floats = 0;
    }
    void* p = nullptr;
    VBQ_CUDA_TRY(dev_alloc(&p, part_floats * sizeof(float)));
    s.part = static_cast<float*>(p);
    s.part_floats = part_floats;
  }
  if (s.n_counters < n_counters) {
    if (s.counters) {
      VBQ_CUDA_TRY(cudaDeviceSynchronize());
      cudaFree(s.counters);
      s.counters = nullptr;
      s.n_counters = 0;
    }
    void* p = nullptr;
    VBQ_CUDA_TRY(dev_alloc(&p, n_counters * sizeof(uint32_t)));
    VBQ_CUDA_TRY(cudaMemset(p, 0, n_counters * sizeof(uint32_t)));
    s.counters = static_cast<uint32_t*>(p);
    s.n_counters = n_counters;
  }
  *out = &s;
  return VBQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vbq_status check_heads(int32_t H, int32_t Hkv, int32_t d, const char* fn) {
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0 || H / Hkv > kAttnMaxGroup)
    return fail(VBQ_ERR_SHAPE, std::string(fn) + ": need H a multiple of H_kv, at most 8 query heads per kv head");
  if (d != 64 && d != 128) return fail(VBQ_ERR_SHAPE, std::string(fn) + ": head_dim must be 64 or 128");
  return VBQ_OK;
}

template <int HD>
vbq_status launch_attn(const AttnArgs& a, int32_t Hkv, cudaStream_t st) {
  static std::once_flag once;
  std::call_once(once, []() {
    cudaFuncSetAttribute(vbq_attn_decode_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         AttnSmem<HD>::kBytes);
  });
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.nparts), static_cast<unsigned>(Hkv), 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = AttnSmem<HD>::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  note_launches(1);
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_attn_decode_kernel<HD>, a));
  return VBQ_OK;
}

}  // namespace

vbq_status launch_attn_prep(const float* qkv, int64_t q_off, int64_t k_off, int64_t v_off, uint16_t* q_rot,
                            uint16_t* k_cache, uint16_t* v_cache, int32_t H, int32_t Hkv, int32_t d, int64_t stride,
                            int32_t pos, double theta, cudaStream_t st) {
  note_launches(1);
  // Programmatic dependent launch: the CTAs start, and compute their angles,
  // as the decode kernel before them drains; they wait for it before reading q, k and v.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(H + Hkv), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(d / 2), 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_attn_prep_kernel, qkv, q_off, k_off, v_off, q_rot, k_cache, v_cache, H, d,
                                  stride, pos, theta));
  return VBQ_OK;
}

}  // namespace vbq

using namespace vbq;

extern "C" vbq_status vbq_rope_append(uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                                      uint16_t* v_cache, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                      int64_t kv_stride, int32_t pos, double theta, void* stream) {
  const vbq_status e = check_heads(n_heads, n_kv_heads, head_dim, "vbq_rope_append");
  if (e != VBQ_OK) return e;
  if (!q || !k_new || !v_new || !k_cache || !v_cache) return fail(VBQ_ERR_INVALID_ARG, "vbq_rope_append: NULL buffer");
  if (pos < 0 || kv_stride <= 0 || pos >= kv_stride)
    return fail(VBQ_ERR_SHAPE, "vbq_rope_append: need 0 <= pos < kv_stride");
  if (!(theta > 1.0)) return fail(VBQ_ERR_INVALID_ARG, "vbq_rope_append: theta must be > 1");
  note_launches(1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(n_heads + n_kv_heads), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(head_dim / 2), 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_rope_append_kernel, q, k_new, v_new, k_cache, v_cache, n_heads,
                                  head_dim, kv_stride, pos, theta));
  return VBQ_OK;
}

extern "C" vbq_status vbq_attention_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                           int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int64_t kv_stride,
                                           int32_t T, float* out, void* stream) {
  const vbq_status e = check_heads(n_heads, n_kv_heads, head_dim, "vbq_attention_decode");
  if (e != VBQ_OK) return e;
  if (!q || !k_cache || !v_cache || !out) return fail(VBQ_ERR_INVALID_ARG, "vbq_attention_decode: NULL buffer");
  if (T < 1 || T > kAttnMaxT || kv_stride < T)
    return fail(VBQ_ERR_SHAPE, "vbq_attention_decode: need 1 <= T <= min(kv_stride, 65536)");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_attention_decode: q and the caches must be 16-byte aligned");
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  int* chk = device_check_word();
  if (!chk) return fail(VBQ_ERR_CUDA, "device check word");
  // Spans: about three CTAs per SM in all, at most kAttnMaxParts per kv head,
  // each a whole number of sub-chunks.
  const int32_t nsub = (T + kAttnSub - 1) / kAttnSub;
  int32_t parts = (gpu_info().sms * 3) / n_kv_heads;
  parts = parts < 1 ? 1 : (parts > kAttnMaxParts ? kAttnMaxParts : parts);
  if (parts > nsub) parts = nsub;
  const int32_t span_sub = (nsub + parts - 1) / parts;
  parts = (nsub + span_sub - 1) / span_sub;
  AttnScratch* s = nullptr;
  const vbq_status se = attn_scratch(dev, static_cast<size_t>(n_kv_heads) * parts * kAttnMaxGroup * part_stride(head_dim),
                                     n_kv_heads, &s);
  if (se != VBQ_OK) return se;
  AttnArgs a{};
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.out = out;
  a.part = s->part;
  a.counters = s->counters;
  a.stride = kv_stride;
  a.T = T;
  a.G = n_heads / n_kv_heads;
  a.nparts = parts;
  a.span = span_sub * kAttnSub;
  a.scale = 1.0f / sqrtf(static_cast<float>(head_dim));
  a.err = chk;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return head_dim == 128 ? launch_attn<128>(a, n_kv_heads, st) : launch_attn<64>(a, n_kv_heads, st);
}
