// Fused dequantize-and-multiply for the packed VBQ layout (layout.h), CUDA cores.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): decode is memory-bound,
// and the packed per-group codes are dequantized and multiplied in one pass.
// The abstract's kernels ran on Apple silicon. This kernel is this library's
// own design for sm_103a:
//
//  * A host-built plan (layout.h) gives each CTA one contiguous, equal-byte
//    range of the packed stream. The range is cut into units at tile borders,
//    and each unit into one slice per warp.
//  * Each warp streams its slices, unit after unit, through a private ring of
//    NSLOT 4 KB slots in shared memory with cp.async.bulk copies completed on
//    mbarriers. The copies start before griddepcontrol.wait, because the packed
//    weights never depend on the previous kernel. Every wait is bounded. The
//    first 512 bytes of each copy into slot 0 are also written past the ring's
//    end, so a record that crosses the end of the ring reads on without
//    wrapping.
//  * The warp walks its slice run by run. A run has one group column g and one
//    bit-class, so each step loop is compiled for its class.
//  * 1-, 2- and 4-bit groups are stored as bit-planes (layout.h), and
//    q - (2^b - 1)/2 = sum_p 2^p (q_p - 1/2). So every lane decodes one 64-bit
//    plane as if it were a 1-bit group, and the b lanes of an entry add their
//    plane sums with weights 2^p.
//  * A plane is decoded with the warp shuffle as a lookup table. Per group
//    column g, lane l holds T_k[l] = sum_{i<5} (bit_i(l) - 1/2) x_{5k+i} for
//    k = 0..12 (the last table covers 4 values). A 5-bit field of the plane
//    selects the lane to read from (shfl.idx uses only the low 5 bits of the
//    lane index), so one shift, one shuffle and one add cover 5 weights.
//  * 8-bit groups keep one byte per code. A byte permute turns code q into the
//    float 1 + q*2^-15, so sum x'_m f_m - C = sum x_m (q_m - 127.5), with
//    x'_m = 2^15 x_m, C = sum (x'_m + 127.5 x_m) per 8-code lane slice, and
//    packed f32x2 FMAs.
//  * Per entry, the lanes of the entry are summed with shuffles, then scaled by
//    the fp16 group scale and added (red.shared.add) into the warp's private
//    fp32 row accumulator. Each warp adds to a row in program order, so the
//    sums do not depend on timing.
//  * Accumulators are double-buffered by unit parity, and no barrier spans the
//    CTA. The last warp to finish a unit (a shared-memory counter) sums the
//    warps' accumulators in warp order while the others go on to the next
//    unit. A tile cut between CTAs gets one partial per unit, and the last CTA
//    to arrive adds them in split order. Results are therefore deterministic.
#pragma once

#include <type_traits>

#include "layout.h"
#include "ptx.cuh"

namespace vbq {

constexpr int CH = 4096;             // bytes per bulk copy and per ring slot
constexpr int LOG_CH = 12;
constexpr int SPILL = 512;           // bytes past the ring's end (>= the largest record, 352 B)
constexpr int XPF = 144;             // floats of activation prep per (warp, column)
constexpr int XP_X = 0, XP_8 = 64, XC_8 = 128;  // x (64), 2^15 x (64), 8-bit slice constants (8)
constexpr int NLUT = 13;             // 5-bit lookup tables per group (the last covers 4 codes)
constexpr int MAX_SEG = 3;

enum XMode : int { X_BF16 = 0, X_RMSNORM = 1, X_GQA = 2, X_SWIGLU = 3 };
enum EpMode : int { EP_STORE = 0, EP_RESID = 1 };

struct MatView {
  const uint8_t* data;
  const uint32_t* run_desc;
  float* y;        // output rows of this matrix, column j at y + j*y_ld
  int32_t y_ld;
  float* trace_y;  // optional raw-output copy (decode-step trace)
};

struct PlanView {
  const UnitRec* units;    // CTA c: slots [c*umax, (c+1)*umax)
  const SliceRec* slices;  // SLICES per slot
  int32_t umax;
  float* partial;          // split-tile partial rows
  uint32_t* counters;      // split-tile arrival counters, zero between launches
};

// Where the activation x (bf16 [NB][K]) comes from.
struct XSource {
  int32_t mode;
  int32_t K;
  const uint16_t* x;  // X_BF16: bf16 [NB][ldx]
  int32_t ldx;
  const float* h;     // X_RMSNORM: fp32 residual [K]
  float eps;
  const float* v;     // X_GQA: fp32 v [n_kv_heads*head_dim]
  int32_t head_dim, group;  // group = n_heads / n_kv_heads
  const float* gate;  // X_SWIGLU: fp32 [K] each
  const float* up;
  uint16_t* trace_x;  // optional: CTA 0 writes the bf16 x it used ([K])
};

struct GemvArgs {
  MatView seg[MAX_SEG];
  int32_t nseg;
  PlanView plan;
  XSource xs;
  int32_t ep;
  const float* resid;  // EP_RESID: y = resid + acc (may alias seg[0].y)
  int* err;
};

template <int NB, int W, int NSLOT>
struct GemvSmem {
  static constexpr int kRingBytes = NSLOT * CH;
  static constexpr int kRingStride = kRingBytes + SPILL;
  static constexpr int kRing = 0;
  static constexpr int kXp = kRing + W * kRingStride;
  static constexpr int kAcc = kXp + W * NB * XPF * 4;          // [2 parities][W][NB][TILE_MAX]
  static constexpr int kAccParity = W * NB * TILE_MAX * 4;
  static constexpr int kBar = kAcc + 2 * kAccParity;
  static constexpr int kMisc = kBar + W * NSLOT * 8;
  static constexpr int kBytes = kMisc + 64 * 4;
  static_assert((kRingBytes & (kRingBytes - 1)) == 0, "ring must be a power of two");
  static_assert(kXp % 64 == 0 && (XPF * 4) % 64 == 0, "prep blocks must be 64-byte aligned");
};

extern __shared__ __align__(1024) uint8_t vbq_smem[];

template <typename T>
__device__ __forceinline__ T lds(uint32_t off) {
  return *reinterpret_cast<const T*>(vbq_smem + off);
}
template <typename T>
__device__ __forceinline__ void sts(uint32_t off, T v) {
  *reinterpret_cast<T*>(vbq_smem + off) = v;
}

// ---- activation values ---------------------------------------------------

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// The inputs from which x[k], x[k+1] (k even) of column col are made.
struct XRaw {
  float a, b, c, d;
};

__device__ __forceinline__ XRaw x_load(const XSource& xs, int col, int k) {
  XRaw r{0.f, 0.f, 0.f, 0.f};
  switch (xs.mode) {
    case X_BF16: {
      const uint32_t v = ldg_nc_u32(xs.x + static_cast<int64_t>(col) * xs.ldx + k);
      r.a = bf16_lo(v);
      r.b = bf16_hi(v);
      break;
    }
    case X_RMSNORM: {
      const float2 h = *reinterpret_cast<const float2*>(xs.h + k);
      r.a = h.x;
      r.b = h.y;
      break;
    }
    case X_GQA: {
      const int head = k / xs.head_dim, j = k - head * xs.head_dim;
      const float2 v = *reinterpret_cast<const float2*>(xs.v + (head / xs.group) * xs.head_dim + j);
      r.a = v.x;
      r.b = v.y;
      break;
    }
    default: {
      const float2 g = *reinterpret_cast<const float2*>(xs.gate + k);
      const float2 u = *reinterpret_cast<const float2*>(xs.up + k);
      r.a = g.x;
      r.b = g.y;
      r.c = u.x;
      r.d = u.y;
      break;
    }
  }
  return r;
}

// x[k], x[k+1] as the bf16 values the projection consumes.
__device__ __forceinline__ float2 x_make(const XSource& xs, const XRaw& r, float inv_rms) {
  switch (xs.mode) {
    case X_BF16: return make_float2(r.a, r.b);
    case X_RMSNORM: return make_float2(round_bf16(r.a * inv_rms), round_bf16(r.b * inv_rms));
    case X_GQA: return make_float2(round_bf16(r.a), round_bf16(r.b));
    default: return make_float2(round_bf16(silu_f(r.a) * r.c), round_bf16(silu_f(r.b) * r.d));
  }
}

// Builds the prep of one column for group g (whole warp; lane owns x_{2l}, x_{2l+1}):
// the 8-bit block in shared memory and this lane's lookup-table registers.
__device__ __forceinline__ void build_prep(uint32_t xp, float x0, float x1, int lane, const float (&sgn)[5],
                                           float (&lut)[NLUT]) {
  sts(xp + (XP_X + 2 * lane) * 4, make_float2(x0, x1));
  const float p0 = x0 * 32768.0f, p1 = x1 * 32768.0f;
  sts(xp + (XP_8 + 2 * lane) * 4, make_float2(p0, p1));
  float c8 = (p0 + p1) + 127.5f * (x0 + x1);
  c8 += __shfl_xor_sync(0xffffffffu, c8, 1);
  c8 += __shfl_xor_sync(0xffffffffu, c8, 2);
  if ((lane & 3) == 0) sts(xp + (XC_8 + (lane >> 2)) * 4, c8);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < NLUT; ++k) lut[k] = 0.0f;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float4 v = lds<float4>(xp + (XP_X + 4 * q) * 4);
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int m = 4 * q + u;
      lut[m / 5] = fmaf(sgn[m % 5], e[u], lut[m / 5]);
    }
  }
}

// ---- decode -------------------------------------------------------------

// One 64-bit plane (w1:w0) against the lookup tables: sum_m (bit_m - 1/2) x_m.
template <int NB>
__device__ __forceinline__ void decode_plane(uint2 cw, const float (&lut)[NB][NLUT], float (&t)[NB]) {
  const uint32_t w0 = cw.x, w1 = cw.y;
  const uint32_t f[NLUT] = {w0,       w0 >> 5,  w0 >> 10, w0 >> 15, w0 >> 20, w0 >> 25, __funnelshift_r(w0, w1, 30),
                            w1 >> 3,  w1 >> 8,  w1 >> 13, w1 >> 18, w1 >> 23, w1 >> 28};
#pragma unroll
  for (int c = 0; c < NB; ++c) {
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < NLUT; ++k) a[k & 3] += __shfl_sync(0xffffffffu, lut[c][k], static_cast<int>(f[k]));
    t[c] = (a[0] + a[1]) + (a[2] + a[3]);
  }
}

// 8-bit entry slice: codes [8*sigma, 8*sigma + 8) in the lane's 8 bytes.
template <int NB>
__device__ __forceinline__ void decode_bytes(uint2 cw, uint32_t xp, uint32_t sigma, float (&t)[NB]) {
  float fv[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    fv[i] = __uint_as_float(__byte_perm(cw.x, 0x3F800000u, 0x7604u | (i << 4)));
    fv[4 + i] = __uint_as_float(__byte_perm(cw.y, 0x3F800000u, 0x7604u | (i << 4)));
  }
  const uint32_t xs = xp + (XP_8 + 8 * sigma) * 4;
#pragma unroll
  for (int c = 0; c < NB; ++c) {
    const float4 xa = lds<float4>(xs + c * XPF * 4);
    const float4 xb = lds<float4>(xs + c * XPF * 4 + 16);
    float2 acc = make_float2(0.0f, 0.0f);
    acc = __ffma2_rn(make_float2(xa.x, xa.y), make_float2(fv[0], fv[1]), acc);
    acc = __ffma2_rn(make_float2(xa.z, xa.w), make_float2(fv[2], fv[3]), acc);
    acc = __ffma2_rn(make_float2(xb.x, xb.y), make_float2(fv[4], fv[5]), acc);
    acc = __ffma2_rn(make_float2(xb.z, xb.w), make_float2(fv[6], fv[7]), acc);
    t[c] = (acc.x + acc.y) - lds<float>(xp + (c * XPF + XC_8 + sigma) * 4);
  }
}

// One step of class CLS with e entries whose record starts at shared offset rb.
// pw = 2^(plane) for the lane's plane (classes 1 and 2).
template <int NB, int CLS>
__device__ __forceinline__ void do_step(uint32_t rb, uint32_t e, uint32_t xp, uint32_t acc, int lane,
                                        const float (&lut)[NB][NLUT], float pw) {
  const uint32_t j = static_cast<uint32_t>(lane) >> CLS;
  const uint32_t sigma = static_cast<uint32_t>(lane) & ((1u << CLS) - 1u);
  const bool active = j < e;
  uint2 cw = make_uint2(0u, 0u);
  if (active) cw = lds<uint2>(rb + 8u * lane);
  float tv[NB];
  if (CLS == 3) {
    decode_bytes<NB>(cw, xp, sigma, tv);
  } else {
    decode_plane<NB>(cw, lut, tv);
    if (CLS > 0) {
#pragma unroll
      for (int c = 0; c < NB; ++c) tv[c] *= pw;
    }
  }
#pragma unroll
  for (int d = 1; d < (1 << CLS); d <<= 1) {
#pragma unroll
    for (int c = 0; c < NB; ++c) tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], d);
  }
  if (active && sigma == 0) {
    const uint16_t sb = lds<uint16_t>(rb + rec_scale_off(CLS, e) + 2u * j);
    const uint32_t row = lds<uint8_t>(rb + rec_row_off(CLS, e) + j);
    const float sc = __half2float(__ushort_as_half(sb));
#pragma unroll
    for (int c = 0; c < NB; ++c)
      atomicAdd(reinterpret_cast<float*>(vbq_smem + acc + (c * TILE_MAX + row) * 4), sc * tv[c]);
  }
}

// Per-warp stream state: the ring, the chunks issued and landed.
struct WarpStream {
  uint32_t ring;      // shared offset of the ring
  uint32_t bar;       // shared address of the first slot's mbarrier
  uint32_t L;         // stream bytes
  uint32_t nch;       // chunks
  uint32_t issued, landed;
  uint32_t avail;     // bytes known to have landed
  uint32_t refill_at; // stream offset at which the next chunk may be issued
  int pu;             // producer: unit being copied
  uint32_t ppos;      // producer: bytes of it already copied
  bool ok;
};

// ---- the kernel ---------------------------------------------------------

template <int NB, int W, int NSLOT>
__global__ void __launch_bounds__(W * 32, 1) vbq_gemv_kernel(const __grid_constant__ GemvArgs a) {
  using Lay = GemvSmem<NB, W, NSLOT>;
  constexpr int SPW = SLICES / W;  // plan slices per warp
  constexpr uint32_t RING = static_cast<uint32_t>(Lay::kRingBytes);
  constexpr uint32_t RMASK = RING - 1u;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int umax = a.plan.umax;

  // Lane i holds unit slot i of this CTA and this warp's slice of it.
  uint32_t u_seg = 0, u_split = 0, u_nsplit = 0, u_pbase = 0, u_cnt = 0, u_r0 = 0, u_rows = 0;
  uint32_t s_run0 = 0, s_k0 = 0, s_run1 = 0, s_k1 = 0, s_b0 = 0, s_b1 = 0, s_g0 = 0;
  if (lane < umax) {
    const size_t slot = static_cast<size_t>(blockIdx.x) * umax + lane;
    const UnitRec ur = a.plan.units[slot];
    u_seg = ur.seg;
    u_split = ur.split;
    u_nsplit = ur.nsplit;
    u_pbase = ur.pbase;
    u_cnt = ur.cnt;
    u_r0 = ur.r0;
    u_rows = ur.rows;
    const SliceRec* sl = a.plan.slices + slot * SLICES + warp * SPW;
    const SliceRec f = sl[0];
    const SliceRec l = sl[SPW - 1];
    s_run0 = f.run0;
    s_k0 = f.k0;
    s_b0 = f.b0;
    s_g0 = f.g0;
    s_run1 = l.run1;
    s_k1 = l.k1;
    s_b1 = l.b1;
    if (SPW > 1 && f.b1 == f.b0) s_g0 = l.g0;  // the first slice is empty
  }
  const int nu = __popc(__ballot_sync(0xffffffffu, u_nsplit > 0u));
  uint32_t len16 = lane < nu ? s_b1 - s_b0 : 0u;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) len16 += __shfl_xor_sync(0xffffffffu, len16, d);

  WarpStream S;
  S.ring = Lay::kRing + warp * Lay::kRingStride;
  S.bar = smem_u32(vbq_smem + Lay::kBar) + warp * NSLOT * 8;
  S.L = len16 * 16u;
  S.nch = (S.L + CH - 1) >> LOG_CH;
  S.issued = S.landed = S.avail = 0;
  S.pu = 0;
  S.ppos = 0;
  S.ok = true;
  const uint32_t ring_a = smem_u32(vbq_smem) + S.ring;
  const uint64_t pol = l2_evict_first_policy();

  auto issue_next = [&]() {  // warp-uniform; lane 0 issues the copies
    const uint32_t slot = S.issued & (NSLOT - 1);
    const uint32_t bytes = min(static_cast<uint32_t>(CH), S.L - S.issued * CH);
    const uint32_t spill = (slot == 0 && S.issued > 0) ? min(static_cast<uint32_t>(SPILL), bytes) : 0u;
    const uint32_t bar = S.bar + 8 * slot;
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes + spill);
    uint32_t done = 0;
    while (done < bytes && S.pu < nu) {
      const uint32_t ub0 = __shfl_sync(0xffffffffu, s_b0, S.pu);
      const uint32_t ub1 = __shfl_sync(0xffffffffu, s_b1, S.pu);
      const uint32_t useg = __shfl_sync(0xffffffffu, u_seg, S.pu);
      const uint32_t ulen = (ub1 - ub0) * 16u;
      const uint32_t take = min(ulen - S.ppos, bytes - done);
      if (take > 0 && lane == 0) {
        const uint8_t* src = a.seg[useg].data + static_cast<uint64_t>(ub0) * 16u + S.ppos;
        bulk_g2s(ring_a + slot * CH + done, src, take, bar, pol);
        if (done < spill) bulk_g2s(ring_a + RING + done, src, min(take, spill - done), bar, pol);
      }
      done += take;
      S.ppos += take;
      if (S.ppos == ulen) {
        ++S.pu;
        S.ppos = 0;
      }
    }
    ++S.issued;
    S.refill_at = S.issued < S.nch ? (S.issued + 1 - NSLOT) * CH : 0xFFFFFFFFu;
  };

  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NSLOT; ++i) mbar_init(S.bar + 8 * i, 1);
    fence_mbarrier_init();
  }
  __syncwarp();
  S.refill_at = 0xFFFFFFFFu;
  while (S.issued < S.nch && S.issued < static_cast<uint32_t>(NSLOT)) issue_next();

  const uint32_t xp = Lay::kXp + warp * NB * XPF * 4;
  float sgn[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) sgn[i] = ((lane >> i) & 1) ? 0.5f : -0.5f;
  const float pw2 = (lane & 1) ? 2.0f : 1.0f;
  const float pw4 = static_cast<float>(1 << (lane & 3));
  float lut[NB][NLUT];
#pragma unroll
  for (int c = 0; c < NB; ++c)
#pragma unroll
    for (int k = 0; k < NLUT; ++k) lut[c][k] = 0.0f;
  // This warp's accumulator for unit parity p: acc_base + p * kAccParity.
  const uint32_t acc_base = Lay::kAcc + warp * NB * TILE_MAX * 4;
  float* misc = reinterpret_cast<float*>(vbq_smem + Lay::kMisc);
  // misc words 32..35: arrivals[2], reductions done[2], as uint32.
  uint32_t* ucount = reinterpret_cast<uint32_t*>(misc) + 32;
  if (threadIdx.x < 4) ucount[threadIdx.x] = 0u;

  __syncthreads();  // the unit counters are initialized

  // The next kernel may start streaming its own weights now.
  grid_dep_launch();
  grid_dep_wait();

  // Start loading x for the first group column before the RMSNorm reduction.
  int pre_g = nu > 0 ? static_cast<int>(__shfl_sync(0xffffffffu, s_g0, 0)) : -1;
  XRaw pre[NB];
  if (pre_g >= 0) {
#pragma unroll
    for (int c = 0; c < NB; ++c) pre[c] = x_load(a.xs, c, pre_g * GROUP + 2 * lane);
  }

  // RMSNorm scale, when the input is rmsnorm(h): every CTA reduces h in the same order.
  float inv_rms = 1.0f;
  if (a.xs.mode == X_RMSNORM) {
    float ss = 0.0f;
    for (int k = threadIdx.x; k < a.xs.K; k += W * 32) {
      const float v = a.xs.h[k];
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) misc[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float tot = 0.0f;
      for (int w = 0; w < W; ++w) tot += misc[w];
      misc[W] = 1.0f / sqrtf(tot / static_cast<float>(a.xs.K) + a.xs.eps);
    }
    __syncthreads();
    inv_rms = misc[W];
  }
  if (a.xs.trace_x && blockIdx.x == 0) {
    for (int k = 2 * threadIdx.x; k < a.xs.K; k += 2 * W * 32) {
      const float2 v = x_make(a.xs, x_load(a.xs, 0, k), inv_rms);
      a.xs.trace_x[k] = bf16_bits(v.x);
      a.xs.trace_x[k + 1] = bf16_bits(v.y);
    }
  }

  uint32_t o = 0;  // stream offset of the next record
  uint32_t acc = acc_base;
  int cur_g = -1;
  int cur_seg = -1;

  // Makes group column g's prep current, and prefetches the inputs of g + 1.
  auto prep_for = [&](int g) {
    XRaw r[NB];
    if (g == pre_g) {
#pragma unroll
      for (int c = 0; c < NB; ++c) r[c] = pre[c];
    } else {
#pragma unroll
      for (int c = 0; c < NB; ++c) r[c] = x_load(a.xs, c, g * GROUP + 2 * lane);
    }
    pre_g = (g + 1) * GROUP < a.xs.K ? g + 1 : -1;
    if (pre_g >= 0) {
#pragma unroll
      for (int c = 0; c < NB; ++c) pre[c] = x_load(a.xs, c, pre_g * GROUP + 2 * lane);
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const float2 xv = x_make(a.xs, r[c], inv_rms);
      build_prep(xp + c * XPF * 4, xv.x, xv.y, lane, sgn, lut[c]);
    }
    __syncwarp();
    cur_g = g;
  };

  // Waits until the bytes below `upto` have landed; false on a timeout.
  auto wait_for = [&](uint32_t upto) {
    while (S.avail < upto) {
      const bool done = mbar_wait(S.bar + 8 * (S.landed & (NSLOT - 1)), (S.landed / NSLOT) & 1u);
      if (!__all_sync(0xffffffffu, done)) {
        S.ok = false;
        return;
      }
      ++S.landed;
      S.avail = min(S.landed * CH, S.L);
    }
  };

  auto refill = [&]() {
    if (o >= S.refill_at) {
      __syncwarp();
      if (lane == 0) fence_proxy_async_smem();
      while (o >= S.refill_at) issue_next();
    }
  };

  // Steps [k, kend) of a run of class CLS with n entries.
  auto run_steps = [&](auto cls_tag, uint32_t k, uint32_t kend, uint32_t n) {
    constexpr int CLS = decltype(cls_tag)::value;
    constexpr uint32_t EPS = entries_per_step(CLS);
    constexpr uint32_t FULL = full_step_bytes(CLS);
    const float pw = CLS == 1 ? pw2 : pw4;
    const uint32_t kfull = min(kend, n / EPS);
    for (; k < kfull; ++k) {
      const uint32_t o1 = o + FULL;
      if (S.avail < o1) {
        wait_for(o1);
        if (!S.ok) return;
      }
      do_step<NB, CLS>(S.ring + (o & RMASK), EPS, xp, acc, lane, lut, pw);
      o = o1;
      refill();
    }
    if (k < kend) {  // the run's last, partial step
      const uint32_t e = n - k * EPS;
      const uint32_t o1 = o + rec_bytes(CLS, e);
      if (S.avail < o1) {
        wait_for(o1);
        if (!S.ok) return;
      }
      do_step<NB, CLS>(S.ring + (o & RMASK), e, xp, acc, lane, lut, pw);
      o = o1;
      refill();
    }
  };

  for (int ui = 0; ui < nu; ++ui) {
    const uint32_t par = static_cast<uint32_t>(ui) & 1u;
    acc = acc_base + par * Lay::kAccParity;
    if (ui >= 2) {  // the reduction of unit ui - 2 must have read this buffer (bounded wait)
      const uint32_t need = static_cast<uint32_t>(ui) >> 1;
      const long long t0 = clock64();
      while (*reinterpret_cast<volatile uint32_t*>(ucount + 2 + par) < need) {
        if (clock64() - t0 > 8000000000LL) {
          S.ok = false;
          break;
        }
      }
      S.ok = __all_sync(0xffffffffu, S.ok);
    }
    for (int i = lane; i < NB * TILE_MAX; i += 32) sts(acc + i * 4, 0.0f);
    __syncwarp();
    const uint32_t seg = __shfl_sync(0xffffffffu, u_seg, ui);
    const uint32_t run1 = __shfl_sync(0xffffffffu, s_run1, ui);
    const uint32_t k1 = __shfl_sync(0xffffffffu, s_k1, ui);
    uint32_t run = __shfl_sync(0xffffffffu, s_run0, ui);
    uint32_t k = __shfl_sync(0xffffffffu, s_k0, ui);
    const uint32_t run_end = run1 + (k1 > 0u ? 1u : 0u);
    const uint32_t* rdesc = a.seg[seg].run_desc;
    if (static_cast<int>(seg) != cur_seg) {
      cur_seg = static_cast<int>(seg);
      cur_g = -1;
    }
    uint32_t dbase = run;
    uint32_t dcur = (run + lane < run_end) ? __ldg(rdesc + run + lane) : 0u;
    uint32_t dnext = (run + 32 + lane < run_end) ? __ldg(rdesc + run + 32 + lane) : 0u;

    for (; S.ok && run < run_end; ++run, k = 0) {
      if (run - dbase >= 32u) {
        dbase += 32;
        dcur = dnext;
        dnext = (dbase + 32 + lane < run_end) ? __ldg(rdesc + dbase + 32 + lane) : 0u;
      }
      const uint32_t d = __shfl_sync(0xffffffffu, dcur, run - dbase);
      const int g = static_cast<int>(run_g(d));
      const uint32_t cls = run_cls(d), n = run_n(d);
      const uint32_t kend = (run == run1) ? k1 : (n + entries_per_step(cls) - 1u) / entries_per_step(cls);
      if (g != cur_g) prep_for(g);
      switch (cls) {
        case 0: run_steps(std::integral_constant<int, 0>{}, k, kend, n); break;
        case 1: run_steps(std::integral_constant<int, 1>{}, k, kend, n); break;
        case 2: run_steps(std::integral_constant<int, 2>{}, k, kend, n); break;
        default: run_steps(std::integral_constant<int, 3>{}, k, kend, n); break;
      }
    }

    // ---- unit epilogue: the last warp to finish sums the warps in fixed order ----
    __syncwarp();
    __threadfence_block();
    uint32_t arrived = 0;
    if (lane == 0) arrived = atomicAdd(ucount + par, 1u);
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived % W == W - 1) {
      __threadfence_block();
      const uint32_t split = __shfl_sync(0xffffffffu, u_split, ui);
      const uint32_t nsplit = __shfl_sync(0xffffffffu, u_nsplit, ui);
      const uint32_t r0 = __shfl_sync(0xffffffffu, u_r0, ui);
      const uint32_t rows = __shfl_sync(0xffffffffu, u_rows, ui);
      const MatView& M = a.seg[seg];
      const uint32_t accp = Lay::kAcc + par * Lay::kAccParity;
      auto store = [&](int c, uint32_t row, float v) {
        if (c == 0 && M.trace_y) M.trace_y[row] = v;
        if (a.ep == EP_RESID) v += a.resid[row];
        M.y[static_cast<int64_t>(c) * M.y_ld + row] = v;
      };
      auto warp_sum = [&](int c, uint32_t r) {
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) v += lds<float>(accp + ((w * NB + c) * TILE_MAX + r) * 4);
        return v;
      };
      if (nsplit <= 1u) {
        for (uint32_t r = lane; r < rows; r += 32) {
#pragma unroll
          for (int c = 0; c < NB; ++c) store(c, r0 + r, warp_sum(c, r));
        }
      } else {
        const uint32_t pbase = __shfl_sync(0xffffffffu, u_pbase, ui);
        const uint32_t cnt = __shfl_sync(0xffffffffu, u_cnt, ui);
        float* part = a.plan.partial + static_cast<size_t>(pbase) * NB;
        for (uint32_t r = lane; r < rows; r += 32) {
#pragma unroll
          for (int c = 0; c < NB; ++c) part[(split * NB + c) * rows + r] = warp_sum(c, r);
        }
        __threadfence();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(a.plan.counters + cnt, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == nsplit - 1u) {
          __threadfence();
          for (uint32_t r = lane; r < rows; r += 32) {
#pragma unroll
            for (int c = 0; c < NB; ++c) {
              float v = 0.0f;
              for (uint32_t s = 0; s < nsplit; ++s) v += __ldcg(part + (s * NB + c) * rows + r);
              store(c, r0 + r, v);
            }
          }
          if (lane == 0) a.plan.counters[cnt] = 0u;
        }
      }
      __syncwarp();
      __threadfence_block();
      if (lane == 0) atomicAdd(ucount + 2 + par, 1u);
    }
  }

  if (!S.ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    // Drain this warp's copies in flight (bounded) before the shared memory is released.
    for (uint32_t c = S.landed; c < S.issued; ++c)
      if (!__all_sync(0xffffffffu, mbar_wait(S.bar + 8 * (c & (NSLOT - 1)), (c / NSLOT) & 1u))) break;
  }
}

}  // namespace vbq
