// Fused dequantize-and-multiply for the packed VBQ layout (layout.h), CUDA cores:
// the single-GEMV kernel and the persistent decode-step kernel.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): decode is memory-bound,
// and the packed per-group codes are dequantized and multiplied in one pass.
// The abstract's kernels ran on Apple silicon. These kernels are this
// library's own design for sm_103a:
//
//  * A host-built plan (plan.h) gives each CTA one contiguous range of the
//    packed stream, balanced by a measured cost model. The range is cut into
//    units at tile borders, and each unit into one slice per warp. Each warp
//    has the list of byte ranges ("pieces") it streams, in order.
//  * Each warp streams its pieces through a private ring of NSLOT 4 KB slots in
//    shared memory with cp.async.bulk copies completed on mbarriers. Every wait
//    is bounded. The first 512 bytes of each copy into slot 0 are also written
//    past the ring's end, so a record that crosses the end of the ring reads on
//    without wrapping. In the decode kernel the pieces of all projections of
//    the step follow each other, so the next projection's weights arrive while
//    the CTAs wait at a grid barrier.
//  * The warp walks its slice run by run. A run has one group column g and one
//    bit class. The step code exists twice, for the three bit-plane classes
//    (their differences are run-time constants) and for bytes: the hot loop
//    must stay small enough for the instruction cache.
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
//  * Per entry, the lanes of the entry are summed with shuffles, scaled by the
//    fp16 group scale and added into the warp's private fp32 row accumulator
//    with a predicated load-add-store (the rows of one group column are
//    distinct, so no atomic is needed). Each warp adds to a row in program
//    order. Full steps whose bytes have landed run two at a time.
//  * Accumulators are double-buffered by unit parity, and no barrier spans the
//    CTA within an item. The last warp to finish a unit sums the warps'
//    accumulators in warp order while the others go on to the next unit (in
//    the decode kernel, the CTA's last unit of an item is summed by all warps
//    together). In the single-GEMV kernel a tile cut between CTAs writes one
//    partial per unit and the last CTA to arrive adds them in split order, so
//    its results are deterministic; the decode kernel adds the partials with
//    fire-and-forget atomics instead.
#pragma once

#include <type_traits>

#include "layout.h"
#include "ptx.cuh"

namespace vbq {

constexpr int CH = 4096;             // bytes per bulk copy and per ring slot
constexpr int LOG_CH = 12;
constexpr int SPILL = 512;           // bytes past the ring's end (>= the largest record, 352 B)
constexpr int XPF = 144;             // floats of activation prep per (warp, column)
// Prep block: x (64), 2^15 x (64) and the 8-bit slice constants (8). 2^15 x is
// stored so that the 8 slices of 8 codes read 128 contiguous bytes per half:
// x'_{8s+t} sits at XP_8 + 4s + t for t < 4 and at XP_8 + 32 + 4s + t - 4 after.
constexpr int XP_X = 0, XP_8 = 64, XC_8 = 128;
constexpr int NLUT = 13;             // 5-bit lookup tables per group (the last covers 4 codes)
constexpr int MAX_SEG = 3;
constexpr uint32_t kNoRefill = 0xFFFFFFFFu;  // WarpStream::refill_at once every chunk is issued
constexpr int XCAP = 16384;          // largest K the decode kernel stages in shared memory

enum XMode : int { X_BF16 = 0, X_RMSNORM = 1, X_GQA = 2, X_SWIGLU = 3 };
enum EpMode : int { EP_STORE = 0, EP_RESID = 1 };

struct MatView {
  const uint8_t* data;
  const uint32_t* run_desc;
  float* y;        // output rows of this matrix, column j at y + j*y_ld (null: the launch's output)
  int64_t y_off;   // when y is null: offset of the output in the launch's output buffer
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
  const uint16_t* x;  // X_BF16: bf16 [NB][ldx] (null: the launch's x)
  int32_t ldx;
  const float* h;     // X_RMSNORM: fp32 residual [K]
  float eps;
  const float* v;     // X_GQA: fp32 v [n_kv_heads*head_dim]
  int32_t head_dim, group;  // group = n_heads / n_kv_heads
  const float* gate;  // X_SWIGLU: fp32 [K] each
  const float* up;
  uint16_t* trace_x;  // optional: CTA 0 writes the bf16 x it used ([K])
};

// A range of floats to clear: ptr + off .. + n (ptr null: the launch's output).
struct ZeroSpec {
  float* ptr;
  int64_t off;
  int32_t n;
};

// A copy of n floats (the decode-step trace of a finished item's output).
struct CopySpec {
  const float* src;
  float* dst;
  int32_t n;
};

// One GEMV over one or more matrices (a "launch item").
struct Item {
  MatView seg[MAX_SEG];
  int32_t nseg;
  PlanView plan;
  XSource xs;
  int32_t ep;
  const float* resid;  // EP_RESID: y = resid + acc (may alias seg[0].y)
  ZeroSpec zero;       // decode kernel: output of the item two later, cleared while this one runs
  CopySpec tcopy;      // decode kernel: trace copy of the previous item's output (trace mode)
};

// A single-item launch: the item plus this plan's per-warp piece lists.
struct GemvArgs {
  Item it;
  const uint64_t* pieces;
  const uint32_t* pstart;  // [n_ctas * W + 1]
  const uint32_t* pbytes;  // [n_ctas * W]
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
  // The decode kernel stages each item's x here (bf16, XCAP values); the
  // single-GEMV kernel reads x from global memory and does not reserve it.
  static constexpr int kX = kBytes;
  static constexpr int kBytesStaged = kX + XCAP * 2;
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

// silu(g) = g / (1 + e^-g) with the fast exponential and division: a few
// 1e-7 of relative error, far below the bf16 rounding that follows.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

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
    // Activations written by another SM earlier in the same launch are read through L2 (ld.cg).
    case X_RMSNORM: {
      const float2 h = __ldcg(reinterpret_cast<const float2*>(xs.h + k));
      r.a = h.x;
      r.b = h.y;
      break;
    }
    case X_GQA: {
      const int head = k / xs.head_dim, j = k - head * xs.head_dim;
      const float2 v = __ldcg(reinterpret_cast<const float2*>(xs.v + (head / xs.group) * xs.head_dim + j));
      r.a = v.x;
      r.b = v.y;
      break;
    }
    default: {
      const float2 g = __ldcg(reinterpret_cast<const float2*>(xs.gate + k));
      const float2 u = __ldcg(reinterpret_cast<const float2*>(xs.up + k));
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
  {
    const int s8 = lane >> 2, t8 = 2 * (lane & 3);  // x_{2l} = x_{8 s8 + t8}
    sts(xp + (XP_8 + (t8 < 4 ? 4 * s8 + t8 : 32 + 4 * s8 + t8 - 4)) * 4, make_float2(p0, p1));
  }
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
  const uint32_t xs = xp + (XP_8 + 4 * sigma) * 4;
#pragma unroll
  for (int c = 0; c < NB; ++c) {
    const float4 xa = lds<float4>(xs + c * XPF * 4);
    const float4 xb = lds<float4>(xs + c * XPF * 4 + 128);
    float2 acc = make_float2(0.0f, 0.0f);
    acc = __ffma2_rn(make_float2(xa.x, xa.y), make_float2(fv[0], fv[1]), acc);
    acc = __ffma2_rn(make_float2(xa.z, xa.w), make_float2(fv[2], fv[3]), acc);
    acc = __ffma2_rn(make_float2(xb.x, xb.y), make_float2(fv[4], fv[5]), acc);
    acc = __ffma2_rn(make_float2(xb.z, xb.w), make_float2(fv[6], fv[7]), acc);
    t[c] = (acc.x + acc.y) - lds<float>(xp + (c * XPF + XC_8 + sigma) * 4);
  }
}

// acc[row] += v in shared memory when p: a predicated load, add and store.
// Not atomic, and it need not be: a warp's accumulators are its own, and the
// entries of one group column have distinct rows, so no two lanes of one
// instruction, nor two steps in flight, touch the same row. (A shared-memory
// fp32 atomic add is a compare-and-swap loop on this GPU.)
__device__ __forceinline__ void acc_add_if(uint32_t addr, float v, bool p) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t.reg .f32 t;\n\tsetp.ne.u32 q, %2, 0;\n\t"
      "@q ld.shared.f32 t, [%0];\n\t@q add.f32 t, t, %1;\n\t@q st.shared.f32 [%0], t;\n\t}" ::"r"(addr),
      "f"(v), "r"(static_cast<uint32_t>(p)));
}

// Decodes one step from its code words and reduces each entry's lanes: on
// return, lane sigma == 0 of entry j holds the entry's dot products. BYTES is
// the 8-bit class; otherwise cls (0, 1 or 2: 1, 2 or 4 bits) is a run-time
// value, so that the three plane classes share one copy of the code (the
// decode loop must stay small enough for the instruction cache).
template <int NB, bool BYTES>
__device__ __forceinline__ void step_dot(uint2 cw, uint32_t xp, uint32_t sigma, uint32_t cls,
                                         const float (&lut)[NB][NLUT], float pw, float (&tv)[NB]) {
  if constexpr (BYTES) {
    decode_bytes<NB>(cw, xp, sigma, tv);
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
#pragma unroll
      for (int c = 0; c < NB; ++c) tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], d);
    }
  } else {
    decode_plane<NB>(cw, lut, tv);
#pragma unroll
    for (int c = 0; c < NB; ++c) tv[c] *= pw;  // 2^plane (1 for 1-bit entries)
    if (cls >= 1u) {
#pragma unroll
      for (int c = 0; c < NB; ++c) tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 1);
    }
    if (cls >= 2u) {
#pragma unroll
      for (int c = 0; c < NB; ++c) tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 2);
    }
  }
}

// U consecutive steps of class CLS, the first at shared offset rb[0], each
// with e entries (e < entries_per_step only for a run's last step). Every lane
// loads and decodes; lanes past the last entry, and all but the first lane of
// an entry, add nothing. The loads of all U steps are issued first.
template <int NB, bool BYTES, int U>
__device__ __forceinline__ void do_steps(const uint32_t (&rb)[U], uint32_t e, uint32_t cls, uint32_t xp,
                                         uint32_t acc, uint32_t acc_a, int lane, const float (&lut)[NB][NLUT],
                                         float pw) {
  if constexpr (BYTES) cls = 3u;
  const uint32_t j = static_cast<uint32_t>(lane) >> cls;
  const uint32_t sigma = static_cast<uint32_t>(lane) & ((1u << cls) - 1u);
  const bool add = j < e && sigma == 0;
  const uint32_t so = rec_scale_off(cls, e) + 2u * j, ro = rec_row_off(cls, e) + j;
  uint2 cw[U];
  uint32_t sb[U], row[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    cw[u] = lds<uint2>(rb[u] + 8u * lane);
    sb[u] = lds<uint16_t>(rb[u] + so);
    row[u] = lds<uint8_t>(rb[u] + ro);
  }
  float tv[U][NB];
#pragma unroll
  for (int u = 0; u < U; ++u) step_dot<NB, BYTES>(cw[u], xp, sigma, cls, lut, pw, tv[u]);
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(sb[u])));
#pragma unroll
    for (int c = 0; c < NB; ++c) acc_add_if(acc_a + (c * TILE_MAX + row[u]) * 4, sc * tv[u][c], add);
  }
  (void)acc;
}

// Stages the x of a decode item in shared memory at sx as the bf16 values the
// projection consumes, for K <= XCAP (K a multiple of 64). All threads of the
// CTA call it; it ends with a CTA barrier. Every CTA computes the same values
// in the same order. Returns the RMSNorm scale (1 for other modes).
template <int W>
__device__ __forceinline__ float stage_x(const XSource& xs, uint32_t sx, float* misc, int lane, int warp) {
  constexpr int NT = W * 32;
  const int K = xs.K;
  const int t = threadIdx.x;
  auto put8 = [&](int k, const float (&v)[8]) {
    uint4 q;
    q.x = bf16_bits(v[0]) | (static_cast<uint32_t>(bf16_bits(v[1])) << 16);
    q.y = bf16_bits(v[2]) | (static_cast<uint32_t>(bf16_bits(v[3])) << 16);
    q.z = bf16_bits(v[4]) | (static_cast<uint32_t>(bf16_bits(v[5])) << 16);
    q.w = bf16_bits(v[6]) | (static_cast<uint32_t>(bf16_bits(v[7])) << 16);
    sts(sx + 2 * k, q);
  };
  auto ld8 = [&](const float* p, float (&v)[8]) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  };
  float inv_rms = 1.0f;
  if (xs.mode == X_RMSNORM) {
    // Pass 1: sum of squares; the first chunk of each thread stays in registers.
    float h0[8];
    float ss = 0.0f;
    const int k0 = 8 * t;
    if (k0 < K) {
      ld8(xs.h + k0, h0);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(h0[i], h0[i], ss);
    }
    for (int k = k0 + 8 * NT; k < K; k += 8 * NT) {
      float v[8];
      ld8(xs.h + k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) misc[warp] = ss;
    __syncthreads();
    if (t == 0) {
      float tot = 0.0f;
      for (int w = 0; w < W; ++w) tot += misc[w];
      misc[W] = 1.0f / sqrtf(tot / static_cast<float>(K) + xs.eps);
    }
    __syncthreads();
    inv_rms = misc[W];
    // Pass 2: bf16(h * inv_rms).
    if (k0 < K) {
#pragma unroll
      for (int i = 0; i < 8; ++i) h0[i] *= inv_rms;
      put8(k0, h0);
    }
    for (int k = k0 + 8 * NT; k < K; k += 8 * NT) {
      float v[8];
      ld8(xs.h + k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] *= inv_rms;
      put8(k, v);
    }
  } else if (xs.mode == X_SWIGLU) {
    // bf16(silu(gate) * up); two chunks of loads in flight per thread.
    for (int k = 8 * t; k < K; k += 16 * NT) {
      const int k2 = k + 8 * NT;
      float g0[8], u0[8], g1[8], u1[8];
      ld8(xs.gate + k, g0);
      ld8(xs.up + k, u0);
      if (k2 < K) {
        ld8(xs.gate + k2, g1);
        ld8(xs.up + k2, u1);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) g0[i] = silu_f(g0[i]) * u0[i];
      put8(k, g0);
      if (k2 < K) {
#pragma unroll
        for (int i = 0; i < 8; ++i) g1[i] = silu_f(g1[i]) * u1[i];
        put8(k2, g1);
      }
    }
  } else if (xs.mode == X_GQA) {
    // bf16(v of the head's kv group), two values at a time (head_dim is even).
#pragma unroll 4
    for (int k = 2 * t; k < K; k += 2 * NT) {
      const int head = k / xs.head_dim, j = k - head * xs.head_dim;
      const float2 v = __ldcg(reinterpret_cast<const float2*>(xs.v + (head / xs.group) * xs.head_dim + j));
      sts(sx + 2 * k, static_cast<uint32_t>(bf16_bits(v.x)) | (static_cast<uint32_t>(bf16_bits(v.y)) << 16));
    }
  } else {  // X_BF16
#pragma unroll 4
    for (int k = 2 * t; k < K; k += 2 * NT) sts(sx + 2 * k, ldg_nc_u32(xs.x + k));
  }
  __syncthreads();
  if (xs.trace_x && blockIdx.x == 0) {
    for (int k = 2 * t; k < K; k += 2 * NT)
      *reinterpret_cast<uint32_t*>(xs.trace_x + k) = lds<uint32_t>(sx + 2 * k);
  }
  return inv_rms;
}

// Per-warp stream of packed bytes: the ring, the chunks issued and landed, and
// the producer's place in the warp's piece list. Lane 0 issues the copies; the
// bookkeeping is warp-uniform.
template <int NSLOT>
struct WarpStream {
  uint32_t ring;       // shared offset of the ring
  uint32_t ring_a;     // shared address of the ring
  uint32_t bar;        // shared address of the first slot's mbarrier
  uint32_t L;          // stream bytes
  uint32_t nch;        // chunks
  uint32_t issued, landed;
  uint32_t avail;      // bytes known to have landed
  uint32_t refill_at;  // stream offset at which the next chunk may be issued
  const uint64_t* pieces;  // this warp's piece list
  uint32_t npieces;
  uint32_t pi;         // producer: piece being copied
  uint32_t ppos;       // producer: bytes of it already copied
  uint64_t pcur, pnext;  // lane i: piece (base + i) and (base + 32 + i) of the list
  uint32_t pbase;      // index of the first piece held in pcur
  uint64_t pol;
  bool ok;

  __device__ __forceinline__ void init(uint32_t ring_off, uint32_t bar_addr, const uint64_t* list, uint32_t n,
                                       uint32_t bytes, int lane) {
    ring = ring_off;
    ring_a = smem_u32(vbq_smem) + ring_off;
    bar = bar_addr;
    L = bytes;
    nch = (bytes + CH - 1) >> LOG_CH;
    issued = landed = avail = 0;
    refill_at = kNoRefill;
    pieces = list;
    npieces = n;
    pi = ppos = 0;
    pbase = 0;
    pcur = lane < static_cast<int>(n) ? __ldg(list + lane) : 0ull;
    pnext = lane + 32 < static_cast<int>(n) ? __ldg(list + 32 + lane) : 0ull;
    pol = l2_evict_first_policy();
    ok = true;
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < NSLOT; ++i) mbar_init(bar + 8 * i, 1);
      fence_mbarrier_init();
    }
    __syncwarp();
  }

  __device__ __forceinline__ void issue_next(int lane) {
    constexpr uint32_t RING = NSLOT * CH;
    const uint32_t slot = issued & (NSLOT - 1);
    const uint32_t bytes = min(static_cast<uint32_t>(CH), L - issued * CH);
    const uint32_t spill = (slot == 0 && issued > 0) ? min(static_cast<uint32_t>(SPILL), bytes) : 0u;
    const uint32_t b = bar + 8 * slot;
    if (lane == 0) mbar_arrive_expect_tx(b, bytes + spill);
    uint32_t done = 0;
    while (done < bytes && pi < npieces) {
      if (pi - pbase >= 32u) {  // next batch of 32 pieces
        pbase += 32;
        pcur = pnext;
        pnext = pbase + 32 + lane < npieces ? __ldg(pieces + pbase + 32 + lane) : 0ull;
      }
      const uint64_t pc = __shfl_sync(0xffffffffu, pcur, static_cast<int>(pi - pbase));
      const uint32_t plen = static_cast<uint32_t>(pc & 0xFFFFFu) << 4;
      const uint32_t take = min(plen - ppos, bytes - done);
      if (lane == 0) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>((pc >> 20) << 4) + ppos;
        bulk_g2s(ring_a + slot * CH + done, src, take, b, pol);
        if (done < spill) bulk_g2s(ring_a + RING + done, src, min(take, spill - done), b, pol);
      }
      done += take;
      ppos += take;
      if (ppos == plen) {
        ++pi;
        ppos = 0;
      }
    }
    ++issued;
    refill_at = issued < nch ? (issued + 1 - NSLOT) * CH : kNoRefill;
  }

  __device__ __forceinline__ void start(int lane) {
    while (issued < nch && issued < static_cast<uint32_t>(NSLOT)) issue_next(lane);
  }

  // Waits until the bytes below `upto` have landed; sets ok = false on a timeout.
  __device__ __forceinline__ void wait_for(uint32_t upto) {
    while (avail < upto) {
      const bool done = mbar_wait(bar + 8 * (landed & (NSLOT - 1)), (landed / NSLOT) & 1u);
      if (!__all_sync(0xffffffffu, done)) {
        ok = false;
        return;
      }
      ++landed;
      avail = min(landed * CH, L);
    }
  }

  // Issues the chunks whose slots the bytes below `o` have freed.
  __device__ __forceinline__ void refill(uint32_t o, int lane) {
    if (o >= refill_at) {
      __syncwarp();
      if (lane == 0) fence_proxy_async_smem();
      while (o >= refill_at) issue_next(lane);
    }
  }

  // After an error: waits (bounded) for the copies still in flight.
  __device__ __forceinline__ void drain() {
    for (uint32_t c = landed; c < issued; ++c)
      if (!__all_sync(0xffffffffu, mbar_wait(bar + 8 * (c & (NSLOT - 1)), (c / NSLOT) & 1u))) break;
  }
};

// Per-warp consumer state that lives across the items of a launch.
template <int NB>
struct Worker {
  uint32_t xp;        // shared offset of this warp's prep block
  uint32_t acc_base;  // shared offset of this warp's accumulators (parity 0)
  float sgn[5];
  float pw2, pw4;
  float lut[NB][NLUT];
  uint32_t o;         // stream offset of the next record
  uint32_t gunit;     // units this CTA has processed, over all items (accumulator parity)
};

// Unit and slice records of one item for this CTA: lane i holds slot i.
struct UnitRegs {
  uint32_t seg, split, nsplit, pbase, cnt, r0, rows;
  uint32_t run0, k0, run1, k1, g0;
};

template <int W>
__device__ __forceinline__ UnitRegs load_units(const PlanView& P, int warp, int lane) {
  constexpr int SPW = SLICES / W;
  UnitRegs u{};
  if (lane < P.umax) {
    const size_t slot = static_cast<size_t>(blockIdx.x) * P.umax + lane;
    const UnitRec ur = P.units[slot];
    u.seg = ur.seg;
    u.split = ur.split;
    u.nsplit = ur.nsplit;
    u.pbase = ur.pbase;
    u.cnt = ur.cnt;
    u.r0 = ur.r0;
    u.rows = ur.rows;
    const SliceRec* sl = P.slices + slot * SLICES + warp * SPW;
    const SliceRec f = sl[0];
    const SliceRec l = sl[SPW - 1];
    u.run0 = f.run0;
    u.k0 = f.k0;
    u.g0 = (SPW > 1 && f.b1 == f.b0) ? l.g0 : f.g0;
    u.run1 = l.run1;
    u.k1 = l.k1;
  }
  return u;
}

// Runs one item for this CTA. All threads of the CTA call it. out/xarg are the
// launch's output and x buffers for matrices and sources that name them.
template <int NB, int W, int NSLOT, bool STAGED>
__device__ __forceinline__ void run_item(const Item& it, const UnitRegs& ur, WarpStream<NSLOT>& S, Worker<NB>& K,
                                         float* out, const uint16_t* xarg, int lane, int warp) {
  static_assert(!STAGED || NB == 1, "staged x is for one column");
  using Lay = GemvSmem<NB, W, NSLOT>;
  constexpr uint32_t RMASK = NSLOT * CH - 1u;
  float* misc = reinterpret_cast<float*>(vbq_smem + Lay::kMisc);
  uint32_t* ucount = reinterpret_cast<uint32_t*>(misc) + 32;
  XSource xs = it.xs;
  if (xs.mode == X_BF16 && xs.x == nullptr) xs.x = xarg;
  const int nu = __popc(__ballot_sync(0xffffffffu, ur.nsplit > 0u));

  // Start loading x for the first group column before the RMSNorm reduction.
  int pre_g = -1;
  XRaw pre[NB];
  float inv_rms = 1.0f;
  if constexpr (STAGED) {
    stage_x<W>(xs, Lay::kX, misc, lane, warp);
  } else {
    pre_g = nu > 0 ? static_cast<int>(__shfl_sync(0xffffffffu, ur.g0, 0)) : -1;
    if (pre_g >= 0) {
#pragma unroll
      for (int c = 0; c < NB; ++c) pre[c] = x_load(xs, c, pre_g * GROUP + 2 * lane);
    }
    // RMSNorm scale, when the input is rmsnorm(h): every CTA reduces h in the same order.
    if (xs.mode == X_RMSNORM) {
      float ss = 0.0f;
      for (int k = threadIdx.x; k < xs.K; k += W * 32) {
        const float v = __ldcg(xs.h + k);
        ss = fmaf(v, v, ss);
      }
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
      if (lane == 0) misc[warp] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float tot = 0.0f;
        for (int w = 0; w < W; ++w) tot += misc[w];
        misc[W] = 1.0f / sqrtf(tot / static_cast<float>(xs.K) + xs.eps);
      }
      __syncthreads();
      inv_rms = misc[W];
    }
    if (xs.trace_x && blockIdx.x == 0) {
      for (int k = 2 * threadIdx.x; k < xs.K; k += 2 * W * 32) {
        const float2 v = x_make(xs, x_load(xs, 0, k), inv_rms);
        xs.trace_x[k] = bf16_bits(v.x);
        xs.trace_x[k + 1] = bf16_bits(v.y);
      }
    }
  }

  int cur_g = -1;
  int cur_seg = -1;
  uint32_t acc = K.acc_base;

  // Makes group column g's prep current, and prefetches the inputs of g + 1.
  auto prep_for = [&](int g) {
    if constexpr (STAGED) {
      const uint32_t v = lds<uint32_t>(Lay::kX + (g * GROUP + 2 * lane) * 2);
      __syncwarp();
      build_prep(K.xp, bf16_lo(v), bf16_hi(v), lane, K.sgn, K.lut[0]);
      __syncwarp();
      cur_g = g;
      return;
    }
    XRaw r[NB];
    if (g == pre_g) {
#pragma unroll
      for (int c = 0; c < NB; ++c) r[c] = pre[c];
    } else {
#pragma unroll
      for (int c = 0; c < NB; ++c) r[c] = x_load(xs, c, g * GROUP + 2 * lane);
    }
    pre_g = (g + 1) * GROUP < xs.K ? g + 1 : -1;
    if (pre_g >= 0) {
#pragma unroll
      for (int c = 0; c < NB; ++c) pre[c] = x_load(xs, c, pre_g * GROUP + 2 * lane);
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const float2 xv = x_make(xs, r[c], inv_rms);
      build_prep(K.xp + c * XPF * 4, xv.x, xv.y, lane, K.sgn, K.lut[c]);
    }
    __syncwarp();
    cur_g = g;
  };

  // Steps [k, kend) of a run of class CLS with n entries. When every byte of
  // the steps has landed (the usual case: a run is about a kilobyte and the
  // ring holds 8), they run with no check at all, in pairs so that two
  // decodes are in flight, and the freed ring slots are refilled after the
  // run. Otherwise full steps go in blocks that need no check inside: every
  // step of a block has landed, and the block ends where the consumed bytes
  // free a ring slot.
  auto run_steps = [&](auto bytes_tag, uint32_t cls, uint32_t k, uint32_t kend, uint32_t n) {
    constexpr bool BYTES = decltype(bytes_tag)::value;
    if constexpr (BYTES) cls = 3u;
    const uint32_t EPS = entries_per_step(cls);
    const uint32_t FULL = full_step_bytes(cls);
    const float pw = cls == 0u ? 1.0f : cls == 1u ? K.pw2 : K.pw4;
    const uint32_t acc_a = smem_u32(vbq_smem) + acc;
    const uint32_t kfull = min(kend, n >> (LOG_STEP_LANES - cls));
    const uint32_t e_last = n - kfull * EPS;  // entries of the partial step, if kend > kfull
    const uint32_t run_end = K.o + (kfull - k) * FULL + (kend > kfull ? rec_bytes(cls, e_last) : 0u);
    const bool landed = run_end <= S.avail;
    while (k < kfull) {
      uint32_t nb = kfull - k;
      if (!landed) {
        if (S.avail < K.o + FULL) {
          S.wait_for(K.o + FULL);
          if (!S.ok) return;
        }
        nb = min(nb, (S.avail - K.o) / FULL);
        if (S.refill_at != kNoRefill) nb = min(nb, (S.refill_at - K.o + FULL - 1u) / FULL);
        if (nb == 0u) {  // cannot happen: refill_at > K.o here; never spin without progress
          S.ok = false;
          return;
        }
      }
      k += nb;
      for (; nb >= 2u; nb -= 2u) {
        const uint32_t rb[2] = {S.ring + (K.o & RMASK), S.ring + ((K.o + FULL) & RMASK)};
        do_steps<NB, BYTES, 2>(rb, EPS, cls, K.xp, acc, acc_a, lane, K.lut, pw);
        K.o += 2u * FULL;
      }
      if (nb) {
        const uint32_t rb[1] = {S.ring + (K.o & RMASK)};
        do_steps<NB, BYTES, 1>(rb, EPS, cls, K.xp, acc, acc_a, lane, K.lut, pw);
        K.o += FULL;
      }
      if (!landed) S.refill(K.o, lane);
    }
    if (S.avail < run_end) {
      S.wait_for(run_end);
      if (!S.ok) return;
    }
    if (kend > kfull) {  // the run's last, partial step
      const uint32_t rb[1] = {S.ring + (K.o & RMASK)};
      do_steps<NB, BYTES, 1>(rb, e_last, cls, K.xp, acc, acc_a, lane, K.lut, pw);
    }
    K.o = run_end;
    S.refill(K.o, lane);
  };

  for (int ui = 0; ui < nu; ++ui, ++K.gunit) {
    const uint32_t par = K.gunit & 1u;
    acc = K.acc_base + par * Lay::kAccParity;
    if (K.gunit >= 2) {  // the reduction of unit gunit - 2 must have read this buffer (bounded wait)
      const uint32_t need = K.gunit >> 1;
      const long long t0 = clock64();
      bool timed_out = false;
      while (*reinterpret_cast<volatile uint32_t*>(ucount + 2 + par) < need) {
        if (clock64() - t0 > kSpinCycles) {
          timed_out = true;
          break;
        }
      }
      if (__any_sync(0xffffffffu, timed_out)) S.ok = false;
    }
    for (int i = lane; i < NB * TILE_MAX; i += 32) sts(acc + i * 4, 0.0f);
    __syncwarp();
    const uint32_t seg = __shfl_sync(0xffffffffu, ur.seg, ui);
    const uint32_t run1 = __shfl_sync(0xffffffffu, ur.run1, ui);
    const uint32_t k1 = __shfl_sync(0xffffffffu, ur.k1, ui);
    uint32_t run = __shfl_sync(0xffffffffu, ur.run0, ui);
    uint32_t k = __shfl_sync(0xffffffffu, ur.k0, ui);
    const uint32_t run_end = run1 + (k1 > 0u ? 1u : 0u);
    const uint32_t* rdesc = it.seg[seg].run_desc;
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
      const uint32_t kend = (run == run1) ? k1 : (n + entries_per_step(cls) - 1u) >> (LOG_STEP_LANES - cls);
      if (g != cur_g) prep_for(g);
      if (cls == 3u) {
        run_steps(std::true_type{}, cls, k, kend, n);
      } else {
        run_steps(std::false_type{}, cls, k, kend, n);
      }
    }

    // ---- unit epilogue: the last warp to finish sums the warps in fixed order ----
    // Every global load of the epilogue is issued before the values are used:
    // it runs while the other SMs stream at full rate, when an L2 round trip
    // takes about a microsecond. In the decode kernel the CTA's last unit of
    // the item is summed after the loop by all warps at once instead, so that
    // no single warp adds the whole tile at the end of the item.
    if (STAGED && ui == nu - 1) continue;
    __syncwarp();
    __threadfence_block();
    uint32_t arrived = 0;
    if (lane == 0) arrived = atomicAdd(ucount + par, 1u);
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived % W == W - 1) {
      __threadfence_block();
      // Rows per lane: 4 lane + j and 128 + 4 lane + j - 4 (j < 8), so that the
      // warp sums read the accumulators 16 bytes at a time without bank conflicts.
      constexpr int RPL = TILE_MAX / 32;
      static_assert(RPL == 8, "the row mapping assumes 256-row tiles");
      const uint32_t split = __shfl_sync(0xffffffffu, ur.split, ui);
      const uint32_t nsplit = __shfl_sync(0xffffffffu, ur.nsplit, ui);
      const uint32_t r0 = __shfl_sync(0xffffffffu, ur.r0, ui);
      const uint32_t rows = __shfl_sync(0xffffffffu, ur.rows, ui);
      const MatView& M = it.seg[seg];
      const uint32_t accp = Lay::kAcc + par * Lay::kAccParity;
      float v[NB][RPL];
#pragma unroll
      for (int c = 0; c < NB; ++c) {
#pragma unroll
        for (int j = 0; j < RPL; ++j) v[c][j] = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) {  // in warp order
          const uint32_t base = accp + ((w * NB + c) * TILE_MAX + 4u * lane) * 4;
          const float4 lo = lds<float4>(base), hi = lds<float4>(base + 128 * 4);
          v[c][0] += lo.x; v[c][1] += lo.y; v[c][2] += lo.z; v[c][3] += lo.w;
          v[c][4] += hi.x; v[c][5] += hi.y; v[c][6] += hi.z; v[c][7] += hi.w;
        }
      }
      // The accumulators are read: let the next unit of this parity have them
      // before any global write (a fence here would wait for those too).
      __syncwarp();
      __threadfence_block();
      if (lane == 0) atomicAdd(ucount + 2 + par, 1u);
      if constexpr (STAGED) {
        // Decode kernel: a whole tile stores its rows, or adds them onto the
        // residual; each split of a tile adds its partial rows into y, which
        // was cleared two items earlier. The adds are fire-and-forget, and the
        // grid barrier after the item makes them visible. The order of the
        // adds of a split tile's partials is not fixed, so those rows can
        // differ in the last bits from one step to the next. (A traced output
        // is added up the same way when the item adds onto the residual, and
        // copied from y by the next item otherwise.)
        float* const ybase = M.y ? M.y : out + M.y_off;
        const bool add = nsplit > 1u || it.ep == EP_RESID;
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          const uint32_t r = (j < 4 ? 4u * lane : 124u + 4u * lane) + j;
          if (r < rows) {
            const float t = v[0][j];
            if (M.trace_y) red_add_f32(M.trace_y + r0 + r, t);
            if (add) {
              red_add_f32(ybase + r0 + r, t);
            } else {
              ybase[r0 + r] = t;
            }
          }
        }
      } else {
        bool mine = true;  // this warp writes the rows
        if (nsplit > 1u) {
          const uint32_t pb = __shfl_sync(0xffffffffu, ur.pbase, ui);
          const uint32_t cnt = __shfl_sync(0xffffffffu, ur.cnt, ui);
          float* part = it.plan.partial + static_cast<size_t>(pb) * NB;
#pragma unroll
          for (int j = 0; j < RPL; ++j) {
            const uint32_t r = (j < 4 ? 4u * lane : 124u + 4u * lane) + j;
#pragma unroll
            for (int c = 0; c < NB; ++c)
              if (r < rows) part[(split * NB + c) * rows + r] = v[c][j];
          }
          __threadfence();
          __syncwarp();
          uint32_t prev = 0;
          if (lane == 0) prev = atomicAdd(it.plan.counters + cnt, 1u);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          mine = prev == nsplit - 1u;
          if (mine) {  // the last split to arrive adds all of them, in split order
            __threadfence();
            constexpr int SB = NB == 1 ? 4 : 1;  // splits whose loads are in flight together
#pragma unroll
            for (int j = 0; j < RPL; ++j)
#pragma unroll
              for (int c = 0; c < NB; ++c) v[c][j] = 0.0f;
            for (uint32_t s0 = 0; s0 < nsplit; s0 += SB) {
              float a[SB][NB][RPL];
#pragma unroll
              for (int q = 0; q < SB; ++q)
#pragma unroll
                for (int j = 0; j < RPL; ++j) {
                  const uint32_t r = (j < 4 ? 4u * lane : 124u + 4u * lane) + j;
#pragma unroll
                  for (int c = 0; c < NB; ++c)
                    a[q][c][j] = (s0 + q < nsplit && r < rows) ? __ldcg(part + ((s0 + q) * NB + c) * rows + r) : 0.0f;
                }
#pragma unroll
              for (int q = 0; q < SB; ++q)
#pragma unroll
                for (int j = 0; j < RPL; ++j)
#pragma unroll
                  for (int c = 0; c < NB; ++c)
                    if (s0 + q < nsplit) v[c][j] += a[q][c][j];
            }
            if (lane == 0) it.plan.counters[cnt] = 0u;
          }
        }
        if (mine) {
          float* const ybase = M.y ? M.y : out + M.y_off;
          float rv[RPL];
#pragma unroll
          for (int j = 0; j < RPL; ++j) {
            const uint32_t r = (j < 4 ? 4u * lane : 124u + 4u * lane) + j;
            rv[j] = (it.ep == EP_RESID && r < rows) ? __ldcg(it.resid + r0 + r) : 0.0f;
          }
#pragma unroll
          for (int j = 0; j < RPL; ++j) {
            const uint32_t r = (j < 4 ? 4u * lane : 124u + 4u * lane) + j;
            if (r < rows) {
#pragma unroll
              for (int c = 0; c < NB; ++c) {
                float t = v[c][j];
                if (c == 0 && M.trace_y) M.trace_y[r0 + r] = t;
                if (it.ep == EP_RESID) t += rv[j];
                ybase[static_cast<int64_t>(c) * M.y_ld + r0 + r] = t;
              }
            }
          }
        }
      }
    }
  }
  if constexpr (STAGED) {
    // The CTA's last unit of the item: warp w sums rows RW w .. RW w + RW - 1
    // (RW = TILE_MAX / W) over the warps' accumulators, in warp order.
    constexpr uint32_t RW = TILE_MAX / W;
    static_assert(!STAGED || (RW <= 32 && RW * W == TILE_MAX), "one lane per row");
    __syncthreads();
    if (nu > 0) {
      const int ui = nu - 1;
      const uint32_t par = (K.gunit - 1u) & 1u;
      const uint32_t seg = __shfl_sync(0xffffffffu, ur.seg, ui);
      const uint32_t nsplit = __shfl_sync(0xffffffffu, ur.nsplit, ui);
      const uint32_t r0 = __shfl_sync(0xffffffffu, ur.r0, ui);
      const uint32_t rows = __shfl_sync(0xffffffffu, ur.rows, ui);
      const MatView& M = it.seg[seg];
      const uint32_t accp = Lay::kAcc + par * Lay::kAccParity;
      const uint32_t r = RW * warp + (lane & (RW - 1u));
      float t = 0.0f;
#pragma unroll
      for (int w = 0; w < W; ++w) t += lds<float>(accp + (w * TILE_MAX + r) * 4);
      // (The next unit of this parity starts after the grid barrier, which
      // orders these reads before its writes; the count only keeps the tally.)
      if (threadIdx.x == 0) atomicAdd(ucount + 2 + par, 1u);
      if (static_cast<uint32_t>(lane) < RW && r < rows) {
        float* const ybase = M.y ? M.y : out + M.y_off;
        if (M.trace_y) red_add_f32(M.trace_y + r0 + r, t);
        if (nsplit > 1u || it.ep == EP_RESID) {
          red_add_f32(ybase + r0 + r, t);
        } else {
          ybase[r0 + r] = t;
        }
      }
    }
  }
}

// Sets up this warp's stream and consumer state.
template <int NB, int W, int NSLOT>
__device__ __forceinline__ void worker_init(WarpStream<NSLOT>& S, Worker<NB>& K, const uint64_t* pieces,
                                            const uint32_t* pstart, const uint32_t* pbytes, int lane, int warp) {
  using Lay = GemvSmem<NB, W, NSLOT>;
  const size_t wi = static_cast<size_t>(blockIdx.x) * W + warp;
  const uint32_t p0 = pstart[wi], p1 = pstart[wi + 1];
  S.init(Lay::kRing + warp * Lay::kRingStride, smem_u32(vbq_smem + Lay::kBar) + warp * NSLOT * 8, pieces + p0,
         p1 - p0, pbytes[wi], lane);
  S.start(lane);
  K.xp = Lay::kXp + warp * NB * XPF * 4;
  K.acc_base = Lay::kAcc + warp * NB * TILE_MAX * 4;
#pragma unroll
  for (int i = 0; i < 5; ++i) K.sgn[i] = ((lane >> i) & 1) ? 0.5f : -0.5f;
  K.pw2 = (lane & 1) ? 2.0f : 1.0f;
  K.pw4 = static_cast<float>(1 << (lane & 3));
#pragma unroll
  for (int c = 0; c < NB; ++c)
#pragma unroll
    for (int k = 0; k < NLUT; ++k) K.lut[c][k] = 0.0f;
  K.o = 0;
  K.gunit = 0;
  uint32_t* ucount = reinterpret_cast<uint32_t*>(vbq_smem + Lay::kMisc) + 32;
  if (threadIdx.x < 4) ucount[threadIdx.x] = 0u;
}

// ---- the single-item kernel ---------------------------------------------

template <int NB, int W, int NSLOT>
__global__ void __launch_bounds__(W * 32, 1) vbq_gemv_kernel(const __grid_constant__ GemvArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WarpStream<NSLOT> S;
  Worker<NB> K;
  const UnitRegs ur = load_units<W>(a.it.plan, warp, lane);
  worker_init<NB, W, NSLOT>(S, K, a.pieces, a.pstart, a.pbytes, lane, warp);
  __syncthreads();  // the unit counters are initialized

  // The next kernel may start streaming its own weights now.
  grid_dep_launch();
  grid_dep_wait();

  run_item<NB, W, NSLOT, false>(a.it, ur, S, K, nullptr, nullptr, lane, warp);
  if (!S.ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    S.drain();
  }
}

// ---- the persistent decode-step kernel ----------------------------------

// A sequence of items with a grid barrier between each and the next. Items
// name their activations by pointer into one workspace; the launch's x and
// output are substituted for items that leave them null.
struct Program {
  const Item* items;
  int32_t n_items;
  const uint64_t* pieces;   // per-warp piece lists over all items
  const uint32_t* pstart;
  const uint32_t* pbytes;
  float* h;                 // h = x is written before the first item
  int32_t d;
  ZeroSpec pre[2];          // outputs of the first two items, cleared before the first barrier
  uint32_t* grid_bar;       // [0]: barrier arrivals, [1]: CTAs done; both zero at launch, and reset at exit
  int* err;
};

struct DecodeArgs {
  Program prog;
  const uint16_t* x;
  float* out;
};

// All threads of the grid copy one range.
__device__ __forceinline__ void grid_copy(const CopySpec& c) {
  if (c.n <= 0) return;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < c.n; i += gridDim.x * blockDim.x)
    c.dst[i] = __ldcg(c.src + i);
}

// All threads of the grid clear one range.
__device__ __forceinline__ void grid_zero(const ZeroSpec& z, float* out) {
  if (z.n <= 0) return;
  float* p = (z.ptr ? z.ptr : out) + z.off;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < z.n; i += gridDim.x * blockDim.x) p[i] = 0.0f;
}

// Grid barrier number k (0-based) of this launch. Bounded: on a timeout it
// records kErrGridTimeout and lets the CTA go on; once any wait has recorded
// an error (the check word is non-zero) it stops waiting at once, so a failed
// step ends in about one wait limit rather than one per barrier.
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

template <int W, int NSLOT>
__global__ void __launch_bounds__(W * 32, 1) vbq_decode_kernel(const __grid_constant__ DecodeArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Program& P = a.prog;
  WarpStream<NSLOT> S;
  Worker<1> K;
  UnitRegs ur = load_units<W>(P.items[0].plan, warp, lane);
  worker_init<1, W, NSLOT>(S, K, P.pieces, P.pstart, P.pbytes, lane, warp);
  // h = x (bf16 -> fp32); the outputs that the first two items add into start at zero.
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < P.d; i += gridDim.x * blockDim.x)
    P.h[i] = __uint_as_float(static_cast<uint32_t>(a.x[i]) << 16);
  grid_zero(P.pre[0], a.out);
  grid_zero(P.pre[1], a.out);
  grid_barrier(P.grid_bar, 0, P.err);
  for (int i = 0; i < P.n_items; ++i) {
    const Item& it = P.items[i];
    grid_zero(it.zero, a.out);
    grid_copy(it.tcopy);
    run_item<1, W, NSLOT, true>(it, ur, S, K, a.out, a.x, lane, warp);
    if (i + 1 < P.n_items) {
      ur = load_units<W>(P.items[i + 1].plan, warp, lane);  // in flight across the barrier
      grid_barrier(P.grid_bar, static_cast<uint32_t>(i + 1), P.err);
    }
  }
  if (!S.ok) {
    if (lane == 0) atomicExch(P.err, kErrRingTimeout);
    S.drain();
  }
  // The last CTA to finish has seen every CTA leave every barrier, so it can
  // return both counters to zero for the next launch in stream order.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(P.grid_bar + 1, 1u) == gridDim.x - 1u) {
      atomicExch(P.grid_bar, 0u);
      atomicExch(P.grid_bar + 1, 0u);
    }
  }
}

}  // namespace vbq
