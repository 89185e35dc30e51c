// The persistent decode-step kernel: every projection of one batch-1 decode
// step in one cooperative launch (one CTA per SM), built from the batch-1
// blocks of gemv.cuh.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): packed per-group codes
// speed up token-by-token decode, which memory bandwidth limits. The pages give
// no architecture; the glue here is this library's reading: unit-gain RMSNorm,
// attention at position 0 (a softmax over one key is 1, so each query head
// returns its kv group's v), SwiGLU, fp32 residual, bf16 projection inputs.
//
// A step is a list of items (one GEMV over one or more matrices) separated by
// grid barriers. At the start of an item every CTA builds the item's input:
//   X_RMS     x = bf16(rmsnorm(h)), h = h_prev + y_add (the previous residual
//             increment); the CTA that owns a 256-value chunk of h writes it
//             to h_next for later items. Every CTA reduces h in the same order.
//   X_GQA     x = bf16(v of each head's kv group), v from [q;k;v].
//   X_SWIGLU  x = bf16(silu(gate) * up), only for the CTA's own columns.
// Outputs are 64-bit fixed-point sums in units of 2^-F_g, F_g per item (stored
// by CTA 0 for the consumers); CTAs accumulate in 32 bits with their own
// exponent F_c and shift at the flush. Every accumulation buffer is cleared by
// a later item once its consumers have read it, so a step leaves them zero.
#pragma once

#include "gemv.cuh"

namespace vbq {

constexpr int XT_MAX = 8192;  // largest K staged whole (RMSNorm and GQA inputs)
constexpr int JT = (XT_MAX + KW * 32 - 1) / (KW * 32);
static_assert(smem_layout(kRingSlots).total + XT_MAX * 2 <= 232448, "shared memory of the decode kernel");

enum XMode : int { X_RMS = 1, X_GQA = 2, X_SWIGLU = 3 };

// A float range filled from fixed-point sums: dst[i] = src[i] * 2^-(*F).
struct CopySpec {
  const unsigned long long* src;
  const int* F;
  float* dst;
  int32_t n;
};

struct ZeroSpec {
  unsigned long long* ptr;
  int64_t n;
};

struct DItem {
  const WarpPlan* warps;     // [n_ctas * KW]
  const CtaPlan* ctas;       // [n_ctas]
  uint32_t seg_st_off[MAX_SEG];
  int32_t mode;
  int32_t K;
  float l1;                  // largest row L1 norm of the item's matrices
  unsigned long long* out;   // fixed-point output in item rows
  int* F_out;                // this item's F_g (written by CTA 0)
  float* maxx_out;           // this item's max |x| (written by CTA 0)
  // X_RMS
  const float* h_prev;       // null: the launch's bf16 x
  const unsigned long long* y_add;  // null: nothing to add
  const int* F_add;
  float* h_next;             // null: not written
  float eps;
  // X_GQA and X_SWIGLU
  const unsigned long long* src;
  const int* F_src;
  int64_t v_off;             // X_GQA: item row of v in src
  int32_t head_dim, group;
  int64_t up_off;            // X_SWIGLU: item row of up in src (gate at row 0)
  const float* maxx_src;     // X_SWIGLU: max |x| of the item that made gate and up
  float l1_gate, l1_up;
  // bookkeeping
  ZeroSpec zero[2];          // buffers cleared during this item
  CopySpec tcopy[3];         // trace: earlier outputs copied out at the start of this item
  uint16_t* trace_x;         // trace: the bf16 input (CTA 0)
};

struct DecodeArgs {
  const DItem* items;
  int32_t n_items;
  const uint64_t* pieces;
  const uint32_t* pstart;
  const uint32_t* pbytes;
  const uint16_t* x;         // bf16 [d]: the step's input
  float* logits;             // [vocab]
  const unsigned long long* logits_acc;  // the head's fixed-point output
  unsigned long long* logits_acc_w;
  const int* F_head;
  int32_t vocab;
  ZeroSpec final_zero;       // cleared after the last item (the head's input increment)
  uint32_t* grid_bar;        // [0]: arrivals, [1]: CTAs done; zero at launch, reset at exit
  int32_t ns;
  int* err;
};

// Grid barrier number k (0-based) of this launch. Bounded: on a timeout it
// records kErrGridTimeout and lets the CTA go on; once any wait has recorded an
// error it stops waiting at once.
__device__ __forceinline__ void grid_barrier(uint32_t* bar, uint32_t k, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint32_t target = (k + 1u) * gridDim.x;
    const long long t0 = clock64();
    uint32_t v;
    int e;
    do {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(e) : "l"(err) : "memory");
      if (e != 0) break;
      if (clock64() - t0 > kSpinCycles) {
        atomicExch(err, kErrGridTimeout);
        break;
      }
    } while (true);
  }
  __syncthreads();
}

__device__ __forceinline__ float fixed_to_float(unsigned long long v, int F) {
  return scalbnf(__ll2float_rn(static_cast<long long>(v)), -F);
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Max over the CTA of a per-thread value (all threads; identical in every CTA for identical inputs).
__device__ __forceinline__ float cta_max(float m, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  __syncthreads();
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < KW; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float cta_sum(float s, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
  __syncthreads();
  if (lane == 0) red[warp] = s;
  __syncthreads();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < KW; ++w) r += red[w];
  return r;
}

// Builds the item's input, stages the CTA's columns and returns (F_c, F_g).
__device__ __forceinline__ int2 stage_item(const DItem& it, const CtaPlan& cp, const SmemLayout& L, uint32_t xt,
                                           const uint16_t* x0, int lane, int warp) {
  float* red = reinterpret_cast<float*>(vbq_smem + L.misc);
  const int K = it.K;
  const uint32_t na = cp.a1 - cp.a0, ncols = na + (cp.b1 - cp.b0);
  const int t = threadIdx.x;
  int Fg = 0;
  float mx_all = 0.0f;
  if (it.mode == X_RMS || it.mode == X_GQA) {
    // The whole input, element k = t + 256 j held by thread t.
    float hv[JT];
    float ss = 0.0f;
    const int F_in = it.mode == X_RMS ? (it.y_add ? *it.F_add : 0) : *it.F_src;
#pragma unroll
    for (int j = 0; j < JT; ++j) {
      const int k = t + j * KW * 32;
      float h = 0.0f;
      if (k < K) {
        if (it.mode == X_RMS) {
          h = it.h_prev ? __ldcg(it.h_prev + k) : __uint_as_float(static_cast<uint32_t>(x0[k]) << 16);
          if (it.y_add) h += fixed_to_float(__ldcg(it.y_add + k), F_in);
        } else {
          const int head = k / it.head_dim, jj = k - head * it.head_dim;
          h = round_bf16(fixed_to_float(__ldcg(it.src + it.v_off + (head / it.group) * it.head_dim + jj), F_in));
        }
      }
      hv[j] = h;
      ss = fmaf(h, h, ss);
    }
    float scale = 1.0f;
    if (it.mode == X_RMS) {
      const float tot = cta_sum(ss, red);
      scale = 1.0f / sqrtf(tot / static_cast<float>(K) + it.eps);
      if (it.h_next) {
#pragma unroll
        for (int j = 0; j < JT; ++j) {
          const int k = t + j * KW * 32;
          if (k < K && static_cast<uint32_t>(k >> 8) % gridDim.x == blockIdx.x) it.h_next[k] = hv[j];
        }
      }
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < JT; ++j) {
      const int k = t + j * KW * 32;
      if (k < K) {
        const uint16_t b = bf16_bits(hv[j] * scale);
        sts<uint16_t>(xt + 2 * k, b);
        m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(b) << 16)));
      }
    }
    mx_all = cta_max(m, red);
    Fg = fixed_exponent(it.l1, mx_all) + 32;
    if (it.trace_x && blockIdx.x == 0)
      for (int k = t; k < K; k += KW * 32) it.trace_x[k] = lds<uint16_t>(xt + 2 * k);
    // Columns of this CTA from the staged input.
    float mc = 0.0f;
    for (uint32_t j = warp; j < ncols; j += KW) {
      const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
      const uint32_t v = lds<uint32_t>(xt + 4 * (g * 32 + lane));
      mc = fmaxf(mc, fmaxf(fabsf(bf16_lo(v)), fabsf(bf16_hi(v))));
    }
    const int Fc = fixed_exponent(it.l1, cta_max(mc, red));
    for (uint32_t j = warp; j < ncols; j += KW) {
      const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
      const uint32_t v = lds<uint32_t>(xt + 4 * (g * 32 + lane));
      put_column(L, static_cast<int>(j), bf16_lo(v), bf16_hi(v), Fc, lane);
    }
    if (blockIdx.x == 0 && t == 0) {
      *it.F_out = Fg;
      *it.maxx_out = mx_all;
    }
    return make_int2(Fc, Fg);
  }
  // X_SWIGLU: only the CTA's columns (at most CCAP / KW per warp), values kept in registers.
  constexpr int CPW = (CCAP + KW - 1) / KW;
  const int F_in = *it.F_src;
  float xv0[CPW], xv1[CPW];
  float mc = 0.0f;
#pragma unroll
  for (int q = 0; q < CPW; ++q) {
    const uint32_t j = warp + q * KW;
    xv0[q] = xv1[q] = 0.0f;
    if (j < ncols) {
      const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
      const int64_t k = static_cast<int64_t>(g) * GROUP + 2 * lane;
      const float g0 = fixed_to_float(__ldcg(it.src + k), F_in), g1 = fixed_to_float(__ldcg(it.src + k + 1), F_in);
      const float u0 = fixed_to_float(__ldcg(it.src + it.up_off + k), F_in);
      const float u1 = fixed_to_float(__ldcg(it.src + it.up_off + k + 1), F_in);
      xv0[q] = round_bf16(silu_f(g0) * u0);
      xv1[q] = round_bf16(silu_f(g1) * u1);
      mc = fmaxf(mc, fmaxf(fabsf(xv0[q]), fabsf(xv1[q])));
    }
  }
  const int Fc = fixed_exponent(it.l1, cta_max(mc, red));
#pragma unroll
  for (int q = 0; q < CPW; ++q) {
    const uint32_t j = warp + q * KW;
    if (j < ncols) put_column(L, static_cast<int>(j), xv0[q], xv1[q], Fc, lane);
  }
  // F_g from a bound: |silu(g)| <= |g| <= l1_gate * max|x_gu|, |up| <= l1_up * max|x_gu|.
  const float mg = *it.maxx_src;
  const float bound = (it.l1_gate * mg) * (it.l1_up * mg);
  Fg = fixed_exponent(it.l1, bound) + 32;
  if (it.trace_x && blockIdx.x == 0) {
    for (int k = t; k < K; k += KW * 32) {
      const float g = fixed_to_float(__ldcg(it.src + k), F_in), u = fixed_to_float(__ldcg(it.src + it.up_off + k), F_in);
      it.trace_x[k] = bf16_bits(silu_f(g) * u);
    }
  }
  if (blockIdx.x == 0 && t == 0) {
    *it.F_out = Fg;
    *it.maxx_out = bound;
  }
  return make_int2(Fc, Fg);
}

// Flush with a shift from the CTA's exponent to the item's: v * 2^(Fg - Fc).
__device__ __forceinline__ void flush_slots_shift(const SmemLayout& L, const CtaPlan& cp, unsigned long long* out,
                                                  int shift) {
  const uint32_t total = cp.n_slots * SROWS;
  for (uint32_t i = threadIdx.x; i < total; i += KW * 32) {
    const int v = lds<int>(L.acc + 4 * i);
    if (v != 0) {
      long long w;
      if (shift >= 0) {
        w = static_cast<long long>(v) << min(shift, 62);
      } else {
        const int r = min(-shift, 62);
        w = (static_cast<long long>(v) + (1ll << (r - 1))) >> r;
      }
      red_add_u64(out + static_cast<size_t>(cp.st_base) * SROWS + i, w);
      sts<int>(L.acc + 4 * i, 0);
    }
  }
}

__global__ void __launch_bounds__(KW * 32, 1) vbq_decode_kernel(const __grid_constant__ DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SmemLayout L = smem_layout(a.ns);
  const uint32_t xt = L.total;  // staged input (bf16 [XT_MAX]) past the batch-1 layout
  WarpStream S;
  Worker K;
  worker_init(S, K, L, static_cast<uint32_t>(a.ns), a.pieces, a.pstart, a.pbytes, lane, warp);
  for (uint32_t i = threadIdx.x; i < SLOTS_MAX * SROWS; i += KW * 32) sts<int>(L.acc + 4 * i, 0);
  __syncthreads();
  for (int ii = 0; ii < a.n_items; ++ii) {
    const DItem& it = a.items[ii];
    const CtaPlan cp = it.ctas[blockIdx.x];
    // Bookkeeping of earlier outputs, spread over the grid.
    const int gt = blockIdx.x * blockDim.x + threadIdx.x, gn = gridDim.x * blockDim.x;
    for (int c = 0; c < 3; ++c) {
      const CopySpec& cs = it.tcopy[c];
      if (cs.n > 0) {
        const int F = *cs.F;
        for (int i = gt; i < cs.n; i += gn) cs.dst[i] = fixed_to_float(__ldcg(cs.src + i), F);
      }
    }
    for (int z = 0; z < 2; ++z)
      for (int64_t i = gt; i < it.zero[z].n; i += gn) it.zero[z].ptr[i] = 0ull;
    const int2 F = stage_item(it, cp, L, xt, a.x, lane, warp);
    K.lut_col = -1;
    __syncthreads();
    if (cp.n_slots > 0) warp_item(L, it.warps + static_cast<size_t>(blockIdx.x) * KW + warp, it.seg_st_off, cp, S, K, lane);
    __syncthreads();
    if (cp.n_slots > 0) flush_slots_shift(L, cp, it.out, F.y - F.x);
    grid_barrier(a.grid_bar, static_cast<uint32_t>(ii), a.err);
  }
  if (!S.ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    S.drain();
  }
  // Logits from the head's fixed-point sums; the sums are cleared for the next step.
  {
    const int F = *a.F_head;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.vocab; i += gridDim.x * blockDim.x) {
      a.logits[i] = fixed_to_float(__ldcg(a.logits_acc + i), F);
      a.logits_acc_w[i] = 0ull;
    }
    for (int64_t i = blockIdx.x * blockDim.x + threadIdx.x; i < a.final_zero.n; i += gridDim.x * blockDim.x)
      a.final_zero.ptr[i] = 0ull;
  }
  // The last CTA to finish has seen every CTA leave every barrier, so it can
  // return both counters to zero for the next launch in stream order.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.grid_bar + 1, 1u) == gridDim.x - 1u) {
      atomicExch(a.grid_bar, 0u);
      atomicExch(a.grid_bar + 1, 0u);
    }
  }
}

}  // namespace vbq
