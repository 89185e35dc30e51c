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
// A step is a list of items (one GEMV over one or more matrices that share an
// input). There is no grid-wide barrier: items are linked by data flow.
//   * Each CTA adds its rows' 32-bit sums into the item's 64-bit fixed-point
//     sums (red.global), then counts itself in on each output super-tile it
//     touched. The CTA that arrives last on a super-tile converts its 1024 rows
//     to float (adding the residual where the item has one), clears the sums,
//     writes the super-tile's (sum of squares, max |value|) for the RMSNorms
//     that read it, and sets the super-tile's flag to the launch's epoch.
//   * A CTA stages an item's input only for its own group columns, after the
//     flags of the super-tiles those columns come from hold the epoch:
//       X_RMS     x = bf16(h * scale), scale = 1 / sqrt(mean(h^2) + eps) from
//                 the residual's per-super-tile statistics (all of them);
//       X_GQA     x = bf16(v of each head's kv group);
//       X_SWIGLU  x = bf16(silu(gate) * up).
//   * The 64-bit sums of an item are in units of 2^-F_g, the same in every CTA:
//     F_g = F + 32 with F from the exact max |x| for X_RMS (monotone rounding:
//     max bf16(|h| * scale) = bf16(max |h| * scale)), else from a bound through
//     the producing item (|v| <= L1 * max|x|, |silu(g) u| <= |g| |u|). Each CTA
//     sums in units of 2^-F_c and shifts by F_g - F_c when it adds in.
// Integer adds do not depend on their order and every float reduction has a
// fixed order, so a step's results do not depend on timing.
#pragma once

#include <stddef.h>

#include "gemv.cuh"

namespace vbq {

constexpr int MAX_RES_SUPER = 8;   // super-tiles of a residual vector (d <= 8192)
constexpr int XT_MAX = MAX_RES_SUPER * SROWS;

enum XMode : int { X_RMS = 1, X_GQA = 2, X_SWIGLU = 3 };

// A residual vector's published statistics: per super-tile (sum of h^2, max |h|) and its flags.
struct ResStats {
  const float2* stats;
  const uint32_t* flag;
  int32_t n_super;
  int32_t K;  // length of the vector
};

struct __align__(16) DItem {
  uint32_t seg_st_off[MAX_SEG];
  int32_t mode;
  int32_t K;                   // input length
  float l1;                    // largest row L1 norm of the item's matrices
  float eps;                   // RMSNorm epsilon
  int32_t n_super;             // item super-tiles
  // output side
  unsigned long long* acc;     // [n_super * SROWS] 64-bit sums, zero between steps
  uint32_t* cnt;               // [n_super] arrivals, zero between steps
  uint32_t* flag;              // [n_super] epoch of the last conversion
  float2* stats;               // [n_super] (sum of squares, max |out|) over rows < out_n, or null
  float* out;                  // float outputs in item rows (null: the launch's logits)
  const float* res;            // residual added to the outputs (item rows), or null
  int64_t out_n;               // rows of out written
  // input side
  const float* src;            // source vector: the residual (X_RMS) or the producing item's outputs
  const uint32_t* src_flag;    // its flags
  int32_t src_nsuper;
  int32_t head_dim, group;     // X_GQA
  ResStats rs;                 // X_RMS: the residual itself; else the residual behind the producer's input
  int64_t v_off;               // X_GQA: item row of v in src
  int32_t v_st0, v_st1;        // X_GQA: v's super-tiles in src
  int64_t up_off;              // X_SWIGLU: item row of up in src (gate at row 0)
  float l1_src;                // X_GQA: L1 bound of the producing item
  float l1_gate, l1_up;        // X_SWIGLU
  // trace (test hooks)
  uint16_t* trace_x;           // the bf16 input, written by CTA 0
  float* trace_y[MAX_SEG];     // per segment: projection outputs before the residual
  int64_t trace_n[MAX_SEG];
};

struct DecodeArgs {
  const DItem* items;
  const CtaPlan* ctas;         // [n_items][gridDim.x]
  const WarpPlan* warps;       // [n_items][gridDim.x][KW]
  int32_t n_items;
  const uint64_t* pieces;
  const uint32_t* pstart;
  const uint32_t* pbytes;
  const uint16_t* x;           // bf16 [d]: the step's input
  int32_t d;
  float* h0;                   // [d] the input as the first residual
  float2* h0_stats;
  uint32_t* h0_flag;
  float* logits;               // [vocab]
  uint32_t epoch;              // this launch's flag value (never 0)
  uint32_t wait_epoch;         // the value waits look for (epoch, except under a test hook)
  long long spin_limit;        // cycles a flag wait may take
  int32_t ns;
  int* err;
};

__device__ __forceinline__ float fixed_to_float(unsigned long long v, int F) {
  return mul_pow2(__ll2float_rn(static_cast<long long>(v)), -F);
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// The e with v < 2^e for v > 0; -300 for 0.
__device__ __forceinline__ int exp_or_floor(float v) { return v > 0.0f ? exp_above(v) : -300; }

// Waits (bounded) until every flag f[0..n) of this lane holds epoch; whole warp.
// Gives up at once if an error is recorded, and records kErrGridTimeout after
// `limit` cycles. Ends with a fence, so the lane's later loads see what was
// written before the flags it polled.
template <int N>
__device__ __forceinline__ void wait_flags(const uint32_t* const (&f)[N], uint32_t epoch, long long limit, int* err) {
  const long long t0 = clock64();
  while (true) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (f[i] && ld_relaxed_u32(f[i]) != epoch) ok = false;
    if (__all_sync(0xffffffffu, ok)) break;
    if (ld_relaxed_s32(err) != 0) break;
    if (clock64() - t0 > limit) {
      atomicExch(err, kErrGridTimeout);
      break;
    }
  }
  fence_acq_rel_gpu();
}

// (scale, max |x|) of x = bf16(h * scale), scale = 1 / sqrt(mean(h^2) + eps),
// from a residual's statistics, summed in super-tile order (the same in every thread).
__device__ __forceinline__ float2 rms_of(const ResStats& rs, float eps) {
  float2 v[MAX_RES_SUPER];
#pragma unroll
  for (int s = 0; s < MAX_RES_SUPER; ++s) v[s] = s < rs.n_super ? __ldcg(rs.stats + s) : make_float2(0.0f, 0.0f);
  float ss = 0.0f, mh = 0.0f;
#pragma unroll
  for (int s = 0; s < MAX_RES_SUPER; ++s) {
    ss += v[s].x;
    mh = fmaxf(mh, v[s].y);
  }
  const float scale = 1.0f / sqrtf(ss / static_cast<float>(rs.K) + eps);
  return make_float2(scale, round_bf16(mh * scale));
}

// The item's fixed-point exponent (CTA sums in units of 2^-F), the same in every CTA.
__device__ __forceinline__ int item_exponent(const DItem& it, float2 r) {
  if (it.mode == X_RMS) return fixed_exponent(it.l1, r.y);
  if (!(r.y > 0.0f) || !(it.l1 > 0.0f)) return 0;
  if (it.mode == X_GQA ? !(it.l1_src > 0.0f) : !(it.l1_gate > 0.0f && it.l1_up > 0.0f)) return 0;
  // Bounds through the producer; one more bit covers its rounding and the bf16 rounding of x.
  const int em = exp_or_floor(r.y);
  if (it.mode == X_GQA) return 30 - (exp_or_floor(it.l1) + exp_or_floor(it.l1_src) + em + 1);
  return 30 - (exp_or_floor(it.l1) + exp_or_floor(it.l1_gate) + exp_or_floor(it.l1_up) + 2 * em + 1);
}

// The source row of input element k (X_GQA).
__device__ __forceinline__ int64_t gqa_row(const DItem& it, uint32_t k) {
  const uint32_t head = k / static_cast<uint32_t>(it.head_dim);
  const uint32_t jj = k - head * static_cast<uint32_t>(it.head_dim);
  return it.v_off + static_cast<int64_t>(head / static_cast<uint32_t>(it.group)) * it.head_dim + jj;
}

// Warp 0 waits (bounded) for the flags of everything the CTA reads for item
// `it`: the residual's statistics, and v (X_GQA) or the gate and up rows of
// each staged column (X_SWIGLU; lane j polls slots j and j + 32). The barrier
// that ends it passes the flags' guarantees to the CTA's other threads. One
// warp per CTA polls, with a short sleep between rounds, so that the polls do
// not crowd the flags' cache lines while the producers write them.
__device__ __forceinline__ void wait_inputs(const DItem& it, const CtaPlan& cp, uint32_t epoch, long long limit,
                                            int* err) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const uint32_t na = cp.a1 - cp.a0, ncols = na + (cp.b1 - cp.b0);
    const uint32_t* f[1 + 4];
    f[0] = lane < it.rs.n_super ? it.rs.flag + lane : nullptr;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t j = static_cast<uint32_t>(lane + 32 * h);
      f[1 + 2 * h] = f[2 + 2 * h] = nullptr;
      if (it.mode == X_RMS || (it.mode == X_SWIGLU && j >= ncols)) continue;
      const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
      const uint32_t k = g * GROUP;
      if (it.mode == X_GQA) {  // all of v's super-tiles (lane j: the j-th and (j + 32)-th)
        const int32_t t = it.v_st0 + lane + 32 * h;
        if (h == 0 && t < it.v_st1) f[1] = it.src_flag + t;
        if (h == 1 && t < it.v_st1) f[3] = it.src_flag + t;
      } else {
        f[1 + 2 * h] = it.src_flag + k / SROWS;
        f[2 + 2 * h] = it.src_flag + (it.up_off + k) / SROWS;
      }
    }
    const long long t0 = clock64();
    while (true) {
      bool ok = true;
#pragma unroll
      for (int i = 0; i < 5; ++i)
        if (f[i] && ld_relaxed_u32(f[i]) != epoch) ok = false;
      if (__all_sync(0xffffffffu, ok)) break;
      if (ld_relaxed_s32(err) != 0) break;
      if (clock64() - t0 > limit) {
        if (lane == 0) atomicExch(err, kErrGridTimeout);
        break;
      }
      __nanosleep(64);
    }
    fence_acq_rel_gpu();  // with the relaxed polls that saw the flags: an acquire
  }
  __syncthreads();
}

// Waits for this CTA's inputs of item `it`, stages its group columns and
// returns (F_c, F_g): the exponent of this CTA's 32-bit sums and the item's
// (the same in every CTA). X_RMS knows the exact max |x|, so F_c = F_g - 32;
// the other modes take F_c from the CTA's own columns (their bound can be
// loose by many bits) at the cost of one barrier. Each warp stages slots
// warp, warp + KW, ...
__device__ __forceinline__ int2 stage_item(const DItem& it, const CtaPlan& cp, const SmemLayout& L, int lane, int warp,
                                          uint32_t epoch, long long limit, int* err) {
  constexpr int CPW = (CCAP + KW - 1) / KW;
  const uint32_t na = cp.a1 - cp.a0, ncols = na + (cp.b1 - cp.b0);
  uint32_t k0[CPW];
  bool has[CPW];
#pragma unroll
  for (int q = 0; q < CPW; ++q) {
    const uint32_t j = static_cast<uint32_t>(warp + q * KW);
    has[q] = j < ncols;
    const uint32_t g = j < na ? cp.a0 + j : cp.b0 + (j - na);
    k0[q] = g * GROUP + 2u * static_cast<uint32_t>(lane);
  }
  int64_t ra[CPW], rb[CPW];
#pragma unroll
  for (int q = 0; q < CPW; ++q) {
    ra[q] = rb[q] = 0;
    if (!has[q] || it.mode == X_RMS) continue;
    if (it.mode == X_GQA) {
      ra[q] = gqa_row(it, k0[q]);
      rb[q] = gqa_row(it, k0[q] + 1);
    } else {
      ra[q] = k0[q];
      rb[q] = it.up_off + k0[q];
    }
  }
  wait_inputs(it, cp, epoch, limit, err);
  const float2 r = rms_of(it.rs, it.eps);
  const int Fi = item_exponent(it, r);
  float x0[CPW], x1[CPW];
  if (it.mode == X_RMS) {
    float2 h[CPW];
#pragma unroll
    for (int q = 0; q < CPW; ++q)
      h[q] = has[q] ? __ldcg(reinterpret_cast<const float2*>(it.src + k0[q])) : make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
      x0[q] = round_bf16(h[q].x * r.x);
      x1[q] = round_bf16(h[q].y * r.x);
    }
  } else if (it.mode == X_GQA) {
    float va[CPW], vb[CPW];
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
      va[q] = has[q] ? __ldcg(it.src + ra[q]) : 0.0f;
      vb[q] = has[q] ? __ldcg(it.src + rb[q]) : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
      x0[q] = round_bf16(va[q]);
      x1[q] = round_bf16(vb[q]);
    }
  } else {
    float2 g[CPW], u[CPW];
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
      g[q] = has[q] ? __ldcg(reinterpret_cast<const float2*>(it.src + ra[q])) : make_float2(0.0f, 0.0f);
      u[q] = has[q] ? __ldcg(reinterpret_cast<const float2*>(it.src + rb[q])) : make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int q = 0; q < CPW; ++q) {
      x0[q] = round_bf16(silu_f(g[q].x) * u[q].x);
      x1[q] = round_bf16(silu_f(g[q].y) * u[q].y);
    }
  }
  int F = Fi;
  if (it.mode != X_RMS) {
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < CPW; ++q) m = fmaxf(m, fmaxf(fabsf(x0[q]), fabsf(x1[q])));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    float* red = reinterpret_cast<float*>(vbq_smem + L.misc);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = 0.0f;
#pragma unroll
    for (int w = 0; w < KW; ++w) m = fmaxf(m, red[w]);
    F = fixed_exponent(it.l1, m);
  }
  if (static_cast<uint32_t>(warp) < ncols) {
    if (ncols <= static_cast<uint32_t>(KW)) {
      const float a[1] = {x0[0]}, b[1] = {x1[0]};
      put_columns<1>(L, warp, KW, ncols, a, b, F, lane);
    } else {
      put_columns<CPW>(L, warp, KW, ncols, x0, x1, F, lane);
    }
  }
  return make_int2(F, Fi + 32);
}

// Trace hook: CTA 0 writes the item's whole bf16 input once all of its source is ready.
__device__ __noinline__ void trace_input(const DItem& it, uint32_t epoch, long long limit, int* err) {
  const uint32_t* f[1];
  for (int s0 = 0; s0 < it.src_nsuper; s0 += 32) {
    const int s = s0 + static_cast<int>(threadIdx.x & 31);
    f[0] = s < it.src_nsuper ? it.src_flag + s : nullptr;
    wait_flags(f, epoch, limit, err);
  }
  __syncthreads();
  __threadfence();
  const float2 r = rms_of(it.rs, it.eps);
  for (int k = threadIdx.x; k < it.K; k += blockDim.x) {
    float x;
    if (it.mode == X_RMS) x = __ldcg(it.src + k) * r.x;
    else if (it.mode == X_GQA) x = __ldcg(it.src + gqa_row(it, k));
    else x = silu_f(__ldcg(it.src + k)) * __ldcg(it.src + it.up_off + k);
    it.trace_x[k] = bf16_bits(x);
  }
}

// Sum and max over the CTA in a fixed order (all threads; thread 0 gets the result).
__device__ __forceinline__ float2 cta_sum_max(float s, float m, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, d);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  }
  if (lane == 0) {
    red[2 * warp] = s;
    red[2 * warp + 1] = m;
  }
  __syncthreads();
  float2 r = make_float2(0.0f, 0.0f);
  if (threadIdx.x == 0)
    for (int w = 0; w < KW; ++w) {
      r.x += red[2 * w];
      r.y = fmaxf(r.y, red[2 * w + 1]);
    }
  return r;
}

// After every thread wrote a super-tile's outputs: its statistics (if wanted) and its flag.
__device__ __forceinline__ void publish(float ss, float mx, float2* stats, uint32_t* flag, uint32_t epoch, float* red) {
  float2 r = make_float2(0.0f, 0.0f);
  if (stats) {
    r = cta_sum_max(ss, mx, red);  // includes a barrier
  } else {
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (stats) *stats = r;
    st_release_u32(flag, epoch);  // cumulative: the CTA's writes, ordered before by the barrier
  }
  __syncthreads();  // red is reused
}

// The last arriver's work on item super-tile st: float outputs, cleared sums, statistics, flag.
__device__ __forceinline__ void convert_super(const DItem& it, uint32_t st, int Fg, float* logits, uint32_t epoch,
                                              float* red) {
  constexpr int NT = KW * 32, PER = SROWS / NT;
  static_assert(SROWS % NT == 0, "rows per thread");
  float* out = it.out ? it.out : logits;
  long long v[PER];
  float rv[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int64_t r = static_cast<int64_t>(st) * SROWS + threadIdx.x + p * NT;
    v[p] = static_cast<long long>(__ldcg(it.acc + r));
    rv[p] = (it.res && r < it.out_n) ? __ldcg(it.res + r) : 0.0f;
  }
  int seg = 0;
#pragma unroll
  for (int s = 1; s < MAX_SEG; ++s)
    if (it.trace_y[s] && st >= it.seg_st_off[s]) seg = s;
  float ss = 0.0f, mx = 0.0f;
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int64_t r = static_cast<int64_t>(st) * SROWS + threadIdx.x + p * NT;
    __stcg(it.acc + r, 0ull);
    const float y = fixed_to_float(static_cast<unsigned long long>(v[p]), Fg);
    if (it.trace_y[seg]) {
      const int64_t lr = r - static_cast<int64_t>(it.seg_st_off[seg]) * SROWS;
      if (lr < it.trace_n[seg]) it.trace_y[seg][lr] = y;
    }
    if (r < it.out_n) {
      const float o = it.res ? rv[p] + y : y;
      out[r] = o;
      ss = fmaf(o, o, ss);
      mx = fmaxf(mx, fabsf(o));
    }
  }
  if (threadIdx.x == 0) it.cnt[st] = 0u;
  publish(ss, mx, it.stats ? it.stats + st : nullptr, it.flag + st, epoch, red);
}

// The step input as the first residual: CTA c converts super-tile c.
__device__ __forceinline__ void convert_input(const DecodeArgs& a, uint32_t c, float* red) {
  constexpr int NT = KW * 32, PER = SROWS / NT;
  float ss = 0.0f, mx = 0.0f;
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int k = static_cast<int>(c) * SROWS + static_cast<int>(threadIdx.x) + p * NT;
    if (k < a.d) {
      const float h = __uint_as_float(static_cast<uint32_t>(a.x[k]) << 16);
      a.h0[k] = h;
      ss = fmaf(h, h, ss);
      mx = fmaxf(mx, fabsf(h));
    }
  }
  publish(ss, mx, a.h0_stats + c, a.h0_flag + c, a.epoch, red);
}

// Shared-memory copy of one item's descriptor and of this CTA's plans.
struct ItemSmem {
  DItem it;
  CtaPlan cp;
  WarpPlan wp[KW];
};
constexpr uint32_t kItemSmem = (sizeof(ItemSmem) + 127u) & ~127u;
static_assert(sizeof(DItem) % 16 == 0 && sizeof(CtaPlan) % 16 == 0 && sizeof(WarpPlan) % 16 == 0, "bulk copies");

// Thread 0: starts copying item ii's descriptor and this CTA's plans into buf.
__device__ __forceinline__ void fetch_item(const DecodeArgs& a, int ii, uint32_t buf, uint32_t bar) {
  const size_t c = static_cast<size_t>(ii) * gridDim.x + blockIdx.x;
  mbar_arrive_expect_tx(bar, sizeof(DItem) + sizeof(CtaPlan) + KW * sizeof(WarpPlan));
  bulk_g2s_plain(buf, a.items + ii, sizeof(DItem), bar);
  bulk_g2s_plain(buf + offsetof(ItemSmem, cp), a.ctas + c, sizeof(CtaPlan), bar);
  bulk_g2s_plain(buf + offsetof(ItemSmem, wp), a.warps + c * KW, KW * sizeof(WarpPlan), bar);
}

// 64-bit sums += this CTA's 32-bit sums * 2^shift (its slots; a negative shift
// rounds to nearest), clearing them.
__device__ __forceinline__ void flush_slots_shift(const SmemLayout& L, const CtaPlan& cp, unsigned long long* acc,
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
      red_add_u64(acc + static_cast<size_t>(cp.st_base) * SROWS + i, w);
      sts<int>(L.acc + 4 * i, 0);
    }
  }
}

__global__ void __launch_bounds__(KW * 32, 1) vbq_decode_kernel(const __grid_constant__ DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const SmemLayout L = smem_layout(a.ns);
  const uint32_t ib = L.total;                              // two ItemSmem buffers
  const uint32_t ibar = smem_u32(vbq_smem) + L.misc + 256;  // their mbarriers
  float* red = reinterpret_cast<float*>(vbq_smem + L.misc);
  uint32_t* fin = reinterpret_cast<uint32_t*>(vbq_smem + L.misc + 192);
  WarpStream S;
  Worker K;
  worker_init(S, K, L, static_cast<uint32_t>(a.ns), a.pieces, a.pstart, a.pbytes, lane, warp);
  for (uint32_t i = threadIdx.x; i < SLOTS_MAX * SROWS; i += KW * 32) sts<int>(L.acc + 4 * i, 0);
  if (threadIdx.x == 0) {
    mbar_init(ibar, 1);
    mbar_init(ibar + 8, 1);
    fence_mbarrier_init();
    fetch_item(a, 0, smem_u32(vbq_smem) + ib, ibar);
  }
  const int n_in = (a.d + SROWS - 1) / SROWS;
  if (static_cast<int>(blockIdx.x) < n_in) convert_input(a, blockIdx.x, red);
  __syncthreads();
  for (int ii = 0; ii < a.n_items; ++ii) {
    const uint32_t buf = ib + (ii & 1) * kItemSmem;
    if (threadIdx.x == 0 && ii + 1 < a.n_items) {
      fence_proxy_async_smem();  // every thread read the buffer's previous contents before the last barrier
      fetch_item(a, ii + 1, smem_u32(vbq_smem) + ib + ((ii + 1) & 1) * kItemSmem, ibar + 8 * ((ii + 1) & 1));
    }
    if (__syncthreads_or(!mbar_wait(ibar + 8 * (ii & 1), (ii >> 1) & 1))) {
      if (threadIdx.x == 0) atomicExch(a.err, kErrGridTimeout);
      break;  // the descriptor never arrived: nothing of this step can be trusted
    }
    const ItemSmem& is = *reinterpret_cast<const ItemSmem*>(vbq_smem + buf);
    const DItem& it = is.it;
    const CtaPlan& cp = is.cp;
    if (it.trace_x && blockIdx.x == 0) trace_input(it, a.wait_epoch, a.spin_limit, a.err);
    if (cp.n_slots > 0) {
      const int2 F = stage_item(it, cp, L, lane, warp, a.wait_epoch, a.spin_limit, a.err);
      K.lut_col = -1;
      __syncthreads();
      warp_item(L, &is.wp[warp], it.seg_st_off, cp, S, K, lane);
      __syncthreads();
      flush_slots_shift(L, cp, it.acc, F.y - F.x);
      __syncthreads();
      if (threadIdx.x == 0) {
        // Release: this CTA's adds (ordered before by the barrier) before its
        // arrival. Acquire: the last arriver sees every other CTA's adds.
        // Both arrivals in flight at once (a CTA touches at most two super-tiles).
        static_assert(SLOTS_MAX == 2, "two arrivals");
        const uint32_t st0 = cp.st_base, st1 = cp.st_base + 1;
        const uint32_t c0 = atom_add_acq_rel_u32(it.cnt + st0, 1u);
        const uint32_t c1 = cp.n_slots > 1 ? atom_add_acq_rel_u32(it.cnt + st1, 1u) : 0u;
        uint32_t nf = 0;
        if (c0 + 1u == cp.expect[0]) fin[1 + nf++] = st0;
        if (cp.n_slots > 1 && c1 + 1u == cp.expect[1]) fin[1 + nf++] = st1;
        fin[0] = nf;
      }
      __syncthreads();
      const uint32_t nf = fin[0];
      for (uint32_t q = 0; q < nf; ++q) convert_super(it, fin[1 + q], F.y, a.logits, a.epoch, red);
    }
    __syncthreads();
  }
  if (!S.ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    S.drain();
  }
}

}  // namespace vbq
