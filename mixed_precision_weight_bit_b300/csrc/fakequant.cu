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
// One warp per group, two weights per lane. Lane b < 4 computes bit-width
// b's scale, reciprocal and mixture weight once for the group; the other
// lanes read them by shuffles. Weights, gradients and outputs stream once.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace vbq {

namespace {

constexpr int kFqWarps = 8;

__device__ __forceinline__ float fq_warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}
__device__ __forceinline__ float fq_warp_max(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

// The group's per-width constants, in every lane: pi_b (mixture weight), s_b
// (step) and r_b (c_b / max|w|); lane b < 4 computes width b's, then shuffles.
struct FqGroup {
  float pi[4], s[4], r[4];
};

__device__ __forceinline__ FqGroup fq_group(const float* alpha, const float* u, int64_t g, float inv_tau, float mx,
                                           int lane) {
  const int k = lane & 3;
  const float qmax = static_cast<float>((1 << (1 << k)) - 1), c = 0.5f * qmax;
  const float z = (alpha[g * 4 + k] - logf(-logf(u[g * 4 + k]))) * inv_tau;
  float m = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const float e = expf(z - m);
  float t = e + __shfl_xor_sync(0xffffffffu, e, 1);
  t = t + __shfl_xor_sync(0xffffffffu, t, 2);
  const float pi = e / t;
  const float sk = mx > 0.0f ? mx / c : 0.0f, rk = mx > 0.0f ? c / mx : 0.0f;
  FqGroup G;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    G.pi[b] = __shfl_sync(0xffffffffu, pi, b);
    G.s[b] = __shfl_sync(0xffffffffu, sk, b);
    G.r[b] = __shfl_sync(0xffffffffu, rk, b);
  }
  return G;
}

// Q_b of the lane's two weights for b = 1, 2, 4, 8 (index 0..3); all zero for an all-zero group.
__device__ __forceinline__ void fq_levels(float w0, float w1, const FqGroup& G, float (&q0)[4], float (&q1)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float qmax = static_cast<float>((1 << (1 << k)) - 1), c = 0.5f * qmax;
    const float a = fminf(fmaxf(rintf(__fadd_rn(__fmul_rn(w0, G.r[k]), c)), 0.0f), qmax);
    const float b = fminf(fmaxf(rintf(__fadd_rn(__fmul_rn(w1, G.r[k]), c)), 0.0f), qmax);
    q0[k] = __fmul_rn(G.s[k], a - c);
    q1[k] = __fmul_rn(G.s[k], b - c);
  }
}

__global__ void __launch_bounds__(kFqWarps * 32) vbq_fq_forward_kernel(const float* __restrict__ W,
                                                                      const float* __restrict__ alpha,
                                                                      const float* __restrict__ u, float inv_tau,
                                                                      int64_t n_groups, float* __restrict__ Wmix) {
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kFqWarps + (threadIdx.x >> 5);
  if (g >= n_groups) return;
  const float2 w = __ldcs(reinterpret_cast<const float2*>(W + g * 64) + lane);
  const float mx = fq_warp_max(fmaxf(fabsf(w.x), fabsf(w.y)));
  const FqGroup P = fq_group(alpha, u, g, inv_tau, mx, lane);
  float q0[4], q1[4];
  fq_levels(w.x, w.y, P, q0, q1);
  float2 o = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o.x = fmaf(P.pi[k], q0[k], o.x);
    o.y = fmaf(P.pi[k], q1[k], o.y);
  }
  __stcs(reinterpret_cast<float2*>(Wmix + g * 64) + lane, o);
}

__global__ void __launch_bounds__(kFqWarps * 32) vbq_fq_backward_kernel(const float* __restrict__ W,
                                                                       const float* __restrict__ alpha,
                                                                       const float* __restrict__ u, float inv_tau,
                                                                       const float* __restrict__ G, int64_t n_groups,
                                                                       float* __restrict__ dW,
                                                                       float* __restrict__ dalpha) {
  const int lane = threadIdx.x & 31;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kFqWarps + (threadIdx.x >> 5);
  if (g >= n_groups) return;
  const float2 w = __ldcs(reinterpret_cast<const float2*>(W + g * 64) + lane);
  const float2 gr = __ldcs(reinterpret_cast<const float2*>(G + g * 64) + lane);
  __stcs(reinterpret_cast<float2*>(dW + g * 64) + lane, gr);  // straight through: sum_b pi_b = 1
  const float mx = fq_warp_max(fmaxf(fabsf(w.x), fabsf(w.y)));
  const FqGroup P = fq_group(alpha, u, g, inv_tau, mx, lane);
  float q0[4], q1[4];
  fq_levels(w.x, w.y, P, q0, q1);
  float D[4], mean = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    D[k] = fq_warp_sum(fmaf(gr.x, q0[k], gr.y * q1[k]));
    mean = fmaf(P.pi[k], D[k], mean);
  }
  if (lane < 4) {
    float d = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k == lane) d = P.pi[k] * inv_tau * (D[k] - mean);
    dalpha[g * 4 + lane] = d;
  }
}

bool fq_aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

vbq_status fq_check(const char* fn, const float* W, const float* alpha, const float* u, float tau, int64_t N,
                    int64_t K) {
  if (N < 0 || K < 0 || K % GROUP) return fail(VBQ_ERR_SHAPE, std::string(fn) + ": need N, K >= 0 and K % 64 == 0");
  if (N * K > 0 && (!W || !alpha || !u)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": NULL buffer");
  if (!(tau > 0.0f)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": tau must be > 0");
  if (!fq_aligned(W)) return fail(VBQ_ERR_INVALID_ARG, std::string(fn) + ": W must be 8-byte aligned");
  return VBQ_OK;
}

unsigned fq_grid(int64_t n_groups) { return static_cast<unsigned>((n_groups + kFqWarps - 1) / kFqWarps); }

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
  if (ng > (int64_t(1) << 40)) return fail(VBQ_ERR_SHAPE, "vbq_fakequant_forward: too many groups");
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
  if (ng > (int64_t(1) << 40)) return fail(VBQ_ERR_SHAPE, "vbq_fakequant_backward: too many groups");
  note_launches(1);
  vbq_fq_backward_kernel<<<fq_grid(ng), kFqWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      W, alpha, u, 1.0f / tau, G, ng, dW, dalpha);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}
