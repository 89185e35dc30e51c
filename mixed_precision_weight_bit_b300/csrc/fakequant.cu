// Training-side fake quantization with a Gumbel-Softmax mixture over the
// bit-widths {1, 2, 4, 8} of every group of 64 weights, and its backward pass
// with the straight-through estimator.
//
// VBQ abstract: the per-group precision is learned by a Gumbel-Softmax
// relaxation over precision logits, optimised alternately with the weights;
// the straight-through estimator carries gradients through the rounding. The
// pages give no formulas, so this is the plainest reading:
//  * Q_b(w) = s_b (q - c_b), c_b = (2^b - 1)/2, s_b = max|w_g| / c_b, and
//    q = rint(w r_b + c_b), r_b = c_b / max|w_g|, clipped to [0, 2^b - 1]
//    (fp32, each operation rounded once, ties to even); Q_b(w) = 0 where the
//    group is all zero;
//  * pi_b = softmax_b((alpha_gb + gumbel_gb) / tau), gumbel = -log(-log u)
//    from uniform u in (0, 1) that the caller draws;
//  * w_mix = sum_b pi_b Q_b(w).
// Backward, for the upstream gradient G = dL/dw_mix: the rounding passes the
// gradient straight through (dQ_b/dw = 1, the scale held constant), so
// dL/dw = G sum_b pi_b = G; and dL/dalpha_b = (pi_b / tau) (D_b - sum_b' pi_b'
// D_b') with D_b = sum_i G_i Q_b(w_i) over the group's weights.
//
// Four groups per warp, eight lanes per group ("octet"), eight weights per
// lane in two 16-byte pieces: lane j of an octet holds weights 4j..4j+3 and
// 32+4j..32+4j+3 of its group, so each of a warp's two loads (and stores)
// covers four whole 128-byte lines. Lane b < 4 of an octet computes
// bit-width b's scale, reciprocal and mixture weight once for the group; the
// other lanes read them by shuffles. An octet past the last group computes on
// zeros (every lane takes part in the shuffles) and stores nothing.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace vbq {

namespace {

constexpr int kFqWarps = 8;
constexpr int kFqGroupsPerWarp = 4;
constexpr int kFqGroupsPerCta = kFqWarps * kFqGroupsPerWarp;

// Reductions over the 8 lanes of an octet.
__device__ __forceinline__ float fq_octet_sum(float v) {
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float fq_octet_max(float v) {
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// The group's per-width constants, in every lane of its octet: pi_b (mixture
// weight), s_b (step) and r_b (c_b / max|w|). Octet lane b < 4 computes width
// b's from a = alpha_gb and uu = u_gb, then shuffles.
struct FqGroup {
  float pi[4], s[4], r[4];
};

__device__ __forceinline__ FqGroup fq_group(float a, float uu, float inv_tau, float mx, int lane) {
  const int k = lane & 3;
  const float qmax = static_cast<float>((1 << (1 << k)) - 1), c = 0.5f * qmax;
  const float z = (a - logf(-logf(uu))) * inv_tau;
  float m = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const float e = expf(z - m);
  float t = e + __shfl_xor_sync(0xffffffffu, e, 1);
  t = t + __shfl_xor_sync(0xffffffffu, t, 2);
  const float pi = e / t;
  const float sk = mx > 0.0f ? mx / c : 0.0f, rk = mx > 0.0f ? c / mx : 0.0f;
  const int base = lane & ~7;
  FqGroup G;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    G.pi[b] = __shfl_sync(0xffffffffu, pi, base + b);
    G.s[b] = __shfl_sync(0xffffffffu, sk, base + b);
    G.r[b] = __shfl_sync(0xffffffffu, rk, base + b);
  }
  return G;
}

// Q_b(w) for b = 1, 2, 4, 8 (index k = 0..3); zero for an all-zero group (r = s = 0).
__device__ __forceinline__ float fq_level(float w, const FqGroup& G, int k) {
  const float qmax = static_cast<float>((1 << (1 << k)) - 1), c = 0.5f * qmax;
  const float q = fminf(fmaxf(rintf(__fadd_rn(__fmul_rn(w, G.r[k]), c)), 0.0f), qmax);
  return __fmul_rn(G.s[k], q - c);
}

// The lane's place: its group, whether that group exists, and the element offsets of its two pieces.
struct FqLane {
  int64_t g;
  bool ok;
  int64_t off0, off1;
};

__device__ __forceinline__ FqLane fq_lane(int64_t n_groups) {
  const int lane = threadIdx.x & 31;
  FqLane L;
  L.g = (static_cast<int64_t>(blockIdx.x) * kFqWarps + (threadIdx.x >> 5)) * kFqGroupsPerWarp + (lane >> 3);
  L.ok = L.g < n_groups;
  L.off0 = L.g * 64 + 4 * (lane & 7);
  L.off1 = L.off0 + 32;
  return L;
}

__device__ __forceinline__ void fq_load8(const float* __restrict__ p, const FqLane& L, float (&v)[8]) {
  float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b = a;
  if (L.ok) {
    a = __ldcs(reinterpret_cast<const float4*>(p + L.off0));
    b = __ldcs(reinterpret_cast<const float4*>(p + L.off1));
  }
  v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
  v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

__device__ __forceinline__ void fq_store8(float* __restrict__ p, const FqLane& L, const float (&v)[8]) {
  if (!L.ok) return;
  __stcs(reinterpret_cast<float4*>(p + L.off0), make_float4(v[0], v[1], v[2], v[3]));
  __stcs(reinterpret_cast<float4*>(p + L.off1), make_float4(v[4], v[5], v[6], v[7]));
}

__device__ __forceinline__ FqGroup fq_group_of(const float* __restrict__ alpha, const float* __restrict__ u,
                                               const FqLane& L, float inv_tau, const float (&w)[8], int lane) {
  const int k = lane & 3;
  const float a = L.ok ? alpha[L.g * 4 + k] : 0.0f;
  const float uu = L.ok ? u[L.g * 4 + k] : 0.5f;
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(w[i]));
  return fq_group(a, uu, inv_tau, fq_octet_max(mx), lane);
}

__global__ void __launch_bounds__(kFqWarps * 32) vbq_fq_forward_kernel(const float* __restrict__ W,
                                                                      const float* __restrict__ alpha,
                                                                      const float* __restrict__ u, float inv_tau,
                                                                      int64_t n_groups, float* __restrict__ Wmix) {
  const int lane = threadIdx.x & 31;
  const FqLane L = fq_lane(n_groups);
  float w[8];
  fq_load8(W, L, w);
  const FqGroup P = fq_group_of(alpha, u, L, inv_tau, w, lane);
  float o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc = fmaf(P.pi[k], fq_level(w[i], P, k), acc);
    o[i] = acc;
  }
  fq_store8(Wmix, L, o);
}

__global__ void __launch_bounds__(kFqWarps * 32) vbq_fq_backward_kernel(const float* __restrict__ W,
                                                                       const float* __restrict__ alpha,
                                                                       const float* __restrict__ u, float inv_tau,
                                                                       const float* __restrict__ G, int64_t n_groups,
                                                                       float* __restrict__ dW,
                                                                       float* __restrict__ dalpha) {
  const int lane = threadIdx.x & 31;
  const FqLane L = fq_lane(n_groups);
  float w[8], gr[8];
  fq_load8(W, L, w);
  fq_load8(G, L, gr);
  fq_store8(dW, L, gr);  // straight through: sum_b pi_b = 1
  const FqGroup P = fq_group_of(alpha, u, L, inv_tau, w, lane);
  float D[4], mean = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(gr[i], fq_level(w[i], P, k), acc);
    D[k] = fq_octet_sum(acc);
    mean = fmaf(P.pi[k], D[k], mean);
  }
  const int sl = lane & 7;
  if (L.ok && sl < 4) {
    float d = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k == sl) d = P.pi[k] * inv_tau * (D[k] - mean);
    dalpha[L.g * 4 + sl] = d;
  }
}

bool fq_aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vbq_status fq_check(const char* fn, const float* W, const float* alpha, const float* u, float tau, int64_t N,
                    int64_t K) {
  if (N < 0 || K < 0 || K % GROUP) return fail(VBQ_ERR_SHAPE, std::string(fn) + ": need N, K >= 0 and K % 64 == 0");
  if (N * K > 0 && (!W || !alpha || !u)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": NULL buffer");
  if (!(tau > 0.0f)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": tau must be > 0");
  if (!fq_aligned(W)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": W must be 16-byte aligned");
  return VBQ_OK;
}

unsigned fq_grid(int64_t n_groups) {
  return static_cast<unsigned>((n_groups + kFqGroupsPerCta - 1) / kFqGroupsPerCta);
}

}  // namespace

}  // namespace vbq

using namespace vbq;

extern "C" vbq_status vbq_fakequant_forward(const float* W, const float* alpha, const float* u, float tau, int64_t N,
                                            int64_t K, float* W_mix, void* stream) {
  vbq_status e = fq_check("vbq_fakequant_forward", W, alpha, u, tau, N, K);
  if (e != VBQ_OK) return e;
  if (N * K == 0) return VBQ_OK;
  if (!W_mix || !fq_aligned(W_mix)) return fail(VBQ_ERR_INVALID_ARG, "vbq_fakequant_forward: W_mix NULL or misaligned");
  const int64_t ng = N * (K / GROUP);
  if (ng > int64_t(0x7fffffff) * kFqGroupsPerCta) return fail(VBQ_ERR_SHAPE, "vbq_fakequant_forward: too many groups");
  note_launches(1);
  vbq_fq_forward_kernel<<<fq_grid(ng), kFqWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(W, alpha, u, 1.0f / tau,
                                                                                              ng, W_mix);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}

extern "C" vbq_status vbq_fakequant_backward(const float* W, const float* alpha, const float* u, float tau,
                                             const float* G, int64_t N, int64_t K, float* dW, float* dalpha,
                                             void* stream) {
  vbq_status e = fq_check("vbq_fakequant_backward", W, alpha, u, tau, N, K);
  if (e != VBQ_OK) return e;
  if (N * K == 0) return VBQ_OK;
  if (!G || !dW || !dalpha || !fq_aligned(G) || !fq_aligned(dW))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_fakequant_backward: G, dW or dalpha NULL or misaligned");
  const int64_t ng = N * (K / GROUP);
  if (ng > int64_t(0x7fffffff) * kFqGroupsPerCta) return fail(VBQ_ERR_SHAPE, "vbq_fakequant_backward: too many groups");
  note_launches(1);
  vbq_fq_backward_kernel<<<fq_grid(ng), kFqWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      W, alpha, u, 1.0f / tau, G, ng, dW, dalpha);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}
