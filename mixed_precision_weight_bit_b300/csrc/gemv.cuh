// Fused dequantize-and-multiply for the packed VBQ layout (layout.h), CUDA cores.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): decode is memory-bound,
// and the packed per-group codes are dequantized and multiplied in one pass.
// The abstract's kernels ran on Apple silicon. This kernel is this library's
// own design for sm_103a:
//
//  * One thread-block cluster per row tile. The C CTAs of the cluster split the
//    tile's step stream evenly, and the warps of a CTA split the CTA's steps.
//  * Each warp streams its contiguous byte range of step records into a private
//    4 KB shared-memory ring with 1 KB cp.async.bulk copies, completed on
//    mbarriers. Every wait is bounded.
//  * Activations: per group column g, each warp builds a "prep" block in shared
//    memory from the 64 values of x in that group:
//      - 1-bit: 16 nibble tables T_j[n] = sum_i (bit_i(n) - 1/2) x_{4j+i}.
//        One lookup covers 4 weights; 16 entries sit in 16 distinct banks, so
//        lookups are conflict-free.
//      - 2/4/8-bit: x'_m = x_m * 2^(8 - f_m*b), where f_m is the field
//        position of code m inside its byte, and C = sum (x'_m + c_b x_m)
//        over each lane slice.
//  * 2/4/8-bit decode: each code byte is shifted to bits 15..22 of a word, and
//    a field at bit p becomes the float 1 + q*2^(p-23) in one LOP3 (OR
//    0x3F800000). Then sum x'_m * f_m - C = sum x_m (q_m - c_b), with packed
//    f32x2 FMAs.
//  * Per entry, the lanes of the entry are summed with shuffles, then scaled by
//    the fp16 group scale and added into the warp's fp32 row accumulator in
//    shared memory. Rows are distinct within a step, so no atomics are needed.
//  * Warps, then the cluster's CTAs (through DSMEM), are summed in a fixed
//    order. Results are deterministic.
#pragma once

#include <cooperative_groups.h>

#include "layout.h"
#include "ptx.cuh"

namespace vbq {

namespace cg = cooperative_groups;

constexpr int RING = 4096;           // bytes per warp
constexpr int CHUNK = 1024;          // bytes per bulk copy
constexpr int NSLOT = RING / CHUNK;  // chunks in flight per warp
constexpr int XPF = 464;             // floats of activation prep per (warp, column)
constexpr int XP_LUT = 0, XP_2 = 256, XP_4 = 320, XP_8 = 384, XC_2 = 448, XC_4 = 450, XC_8 = 454;
constexpr int MAX_SEG = 3;

enum XMode : int { X_BF16 = 0, X_RMSNORM = 1, X_GQA = 2, X_SWIGLU = 3 };
enum EpMode : int { EP_STORE = 0, EP_RESID = 1 };

struct MatView {
  const uint8_t* data;
  const uint32_t* desc;
  const uint32_t* off;
  const uint32_t* row0;
  const uint32_t* step0;
  int32_t n_tiles;
  int32_t N;
  float* y;        // output rows of this segment, column j at y + j*y_ld
  int32_t y_ld;
  float* trace_y;  // optional raw-output copy (decode-step trace)
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
  int32_t tile_base[MAX_SEG + 1];  // cumulative tiles: segment s owns [tile_base[s], tile_base[s+1])
  XSource xs;
  int32_t ep;
  const float* resid;  // EP_RESID: y = resid + acc (may alias seg[0].y)
  int* err;
};

template <int NB, int NWARPS>
struct GemvSmem {
  static constexpr int kRing = 0;
  static constexpr int kXp = kRing + NWARPS * RING;
  static constexpr int kAcc = kXp + NWARPS * NB * XPF * 4;
  static constexpr int kPart = kAcc + NWARPS * NB * TILE_MAX * 4;
  static constexpr int kBar = kPart + NB * TILE_MAX * 4;
  static constexpr int kMisc = kBar + NWARPS * NSLOT * 8;
  static constexpr int kBytes = kMisc + 64;
};

// ---- activation values ---------------------------------------------------

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// x[k], x[k+1] (k even) of batch column col, as the bf16 values the projection consumes.
__device__ __forceinline__ float2 x_pair(const XSource& xs, int col, int k, float inv_rms) {
  switch (xs.mode) {
    case X_BF16: {
      const uint32_t v = ldg_nc_u32(xs.x + static_cast<int64_t>(col) * xs.ldx + k);
      return make_float2(bf16_lo(v), bf16_hi(v));
    }
    case X_RMSNORM: {
      const float2 h = *reinterpret_cast<const float2*>(xs.h + k);
      return make_float2(round_bf16(h.x * inv_rms), round_bf16(h.y * inv_rms));
    }
    case X_GQA: {
      const int head = k / xs.head_dim, j = k - head * xs.head_dim;
      const float2 v = *reinterpret_cast<const float2*>(xs.v + (head / xs.group) * xs.head_dim + j);
      return make_float2(round_bf16(v.x), round_bf16(v.y));
    }
    default: {
      const float2 g = *reinterpret_cast<const float2*>(xs.gate + k);
      const float2 u = *reinterpret_cast<const float2*>(xs.up + k);
      return make_float2(round_bf16(silu_f(g.x) * u.x), round_bf16(silu_f(g.y) * u.y));
    }
  }
}

// Builds the prep block of one column for group g (whole warp; lane owns x_{2l}, x_{2l+1}).
__device__ __forceinline__ void build_prep(float* xp, float x0, float x1, int lane) {
  // 1-bit nibble tables: lane covers table j = lane/2, entries n = 8h..8h+7.
  const int j = lane >> 1, h = lane & 1;
  const float a0 = __shfl_sync(0xffffffffu, x0, 2 * j), a1 = __shfl_sync(0xffffffffu, x1, 2 * j);
  const float a2 = __shfl_sync(0xffffffffu, x0, 2 * j + 1), a3 = __shfl_sync(0xffffffffu, x1, 2 * j + 1);
  const float s3 = h ? a3 : -a3;
  float t[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    t[k] = 0.5f * ((((k & 1) ? a0 : -a0) + ((k & 2) ? a1 : -a1)) + ((k & 4) ? a2 : -a2) + s3);
  float4* dst = reinterpret_cast<float4*>(xp + XP_LUT + 16 * j + 8 * h);
  dst[0] = make_float4(t[0], t[1], t[2], t[3]);
  dst[1] = make_float4(t[4], t[5], t[6], t[7]);
  // Pre-scaled copies for the 2/4/8-bit decode: field f of code m gets 2^(8 - f*b).
  const float f2a = (lane & 1) ? 16.0f : 256.0f, f2b = (lane & 1) ? 4.0f : 64.0f;
  const float p2a = x0 * f2a, p2b = x1 * f2b;
  const float p4a = x0 * 256.0f, p4b = x1 * 16.0f;
  const float p8a = x0 * 256.0f, p8b = x1 * 256.0f;
  reinterpret_cast<float2*>(xp + XP_2)[lane] = make_float2(p2a, p2b);
  reinterpret_cast<float2*>(xp + XP_4)[lane] = make_float2(p4a, p4b);
  reinterpret_cast<float2*>(xp + XP_8)[lane] = make_float2(p8a, p8b);
  // Slice constants C = sum over the slice of (x'_m + c_b x_m).
  const float xs = x0 + x1;
  float c2 = (p2a + p2b) + 1.5f * xs;
  float c4 = (p4a + p4b) + 7.5f * xs;
  float c8 = (p8a + p8b) + 127.5f * xs;
#pragma unroll
  for (int d = 1; d < 16; d <<= 1) c2 += __shfl_xor_sync(0xffffffffu, c2, d);
#pragma unroll
  for (int d = 1; d < 8; d <<= 1) c4 += __shfl_xor_sync(0xffffffffu, c4, d);
#pragma unroll
  for (int d = 1; d < 4; d <<= 1) c8 += __shfl_xor_sync(0xffffffffu, c8, d);
  if ((lane & 15) == 0) xp[XC_2 + (lane >> 4)] = c2;
  if ((lane & 7) == 0) xp[XC_4 + (lane >> 3)] = c4;
  if ((lane & 3) == 0) xp[XC_8 + (lane >> 2)] = c8;
}

// ---- decode -------------------------------------------------------------

// 1-bit entry: sum over 16 nibbles of T_j[nibble_j] = sum_m (q_m - 1/2) x_m.
template <int NB>
__device__ __forceinline__ void decode_lut(uint2 cw, uint32_t xp_addr, float (&t)[NB]) {
  float a[NB][4];
#pragma unroll
  for (int c = 0; c < NB; ++c) a[c][0] = a[c][1] = a[c][2] = a[c][3] = 0.0f;
#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    const uint32_t w = wi ? cw.y : cw.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t nib4 = (i == 0) ? (w << 2) : (w >> (4 * i - 2));
      const uint32_t addr = (nib4 & 0x3Cu) | xp_addr;  // xp_addr is 64-byte aligned
#pragma unroll
      for (int c = 0; c < NB; ++c) a[c][i & 3] += lds_f32(addr + c * XPF * 4 + (wi * 8 + i) * 64);
    }
  }
#pragma unroll
  for (int c = 0; c < NB; ++c) t[c] = (a[c][0] + a[c][1]) + (a[c][2] + a[c][3]);
}

// b-bit entry slice (b = 2, 4, 8): 64/b codes in the lane's 8 bytes.
template <int NB, int BITS>
__device__ __forceinline__ void decode_direct(uint2 cw, const float* xp, uint32_t sigma, float (&t)[NB]) {
  constexpr int F = 8 / BITS;       // fields per byte
  constexpr int NPER = 64 / BITS;   // codes per slice
  constexpr uint32_t MK = (1u << BITS) - 1u;
  constexpr int XOFF = BITS == 2 ? XP_2 : BITS == 4 ? XP_4 : XP_8;
  constexpr int COFF = BITS == 2 ? XC_2 : BITS == 4 ? XC_4 : XC_8;
  float fv[NPER];
#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    const uint32_t w = wi ? cw.y : cw.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t S = (i == 0) ? (w << 15) : (i == 1) ? (w << 7) : (i == 2) ? (w >> 1) : (w >> 9);
#pragma unroll
      for (int f = 0; f < F; ++f)
        fv[(wi * 4 + i) * F + f] = __uint_as_float((S & (MK << (15 + f * BITS))) | 0x3F800000u);
    }
  }
#pragma unroll
  for (int c = 0; c < NB; ++c) {
    const float4* xs = reinterpret_cast<const float4*>(xp + c * XPF + XOFF + sigma * NPER);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int p = 0; p < NPER / 4; ++p) {
      const float4 xv = xs[p];
      acc = __ffma2_rn(make_float2(xv.x, xv.y), make_float2(fv[4 * p], fv[4 * p + 1]), acc);
      acc = __ffma2_rn(make_float2(xv.z, xv.w), make_float2(fv[4 * p + 2], fv[4 * p + 3]), acc);
    }
    t[c] = (acc.x + acc.y) - xp[c * XPF + COFF + sigma];
  }
}

// ---- the kernel ---------------------------------------------------------

template <int NB, int NWARPS>
__global__ void __launch_bounds__(NWARPS * 32) vbq_gemv_kernel(const __grid_constant__ GemvArgs a) {
  using L = GemvSmem<NB, NWARPS>;
  extern __shared__ __align__(1024) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tglob = blockIdx.x / C;

  int sidx = 0;
#pragma unroll
  for (int s = 1; s < MAX_SEG; ++s)
    if (s < a.nseg && tglob >= a.tile_base[s]) sidx = s;
  const MatView& M = a.seg[sidx];
  const int t = tglob - a.tile_base[sidx];
  const uint32_t r0 = M.row0[t], rows = M.row0[t + 1] - r0;
  const uint32_t s0 = M.step0[t], ns = M.step0[t + 1] - s0;
  const uint32_t ca = s0 + static_cast<uint32_t>((static_cast<uint64_t>(ns) * rank) / C);
  const uint32_t cb = s0 + static_cast<uint32_t>((static_cast<uint64_t>(ns) * (rank + 1)) / C);
  const uint32_t wa = ca + static_cast<uint32_t>((static_cast<uint64_t>(cb - ca) * warp) / NWARPS);
  const uint32_t wb = ca + static_cast<uint32_t>((static_cast<uint64_t>(cb - ca) * (warp + 1)) / NWARPS);

  uint8_t* ring = smem + L::kRing + warp * RING;
  const uint32_t ring_a = smem_u32(ring);
  float* xp = reinterpret_cast<float*>(smem + L::kXp) + warp * NB * XPF;
  const uint32_t xp_a = smem_u32(xp);
  float* acc = reinterpret_cast<float*>(smem + L::kAcc) + warp * NB * TILE_MAX;
  float* part = reinterpret_cast<float*>(smem + L::kPart);
  const uint32_t bar_a = smem_u32(smem + L::kBar) + warp * NSLOT * 8;
  float* misc = reinterpret_cast<float*>(smem + L::kMisc);

  // Start streaming this warp's weights before waiting on the previous kernel:
  // the packed weights never depend on it.
  const uint64_t gbase = static_cast<uint64_t>(M.off[wa]) * 16u;
  const uint32_t len = static_cast<uint32_t>(static_cast<uint64_t>(M.off[wb]) * 16u - gbase);
  const uint32_t nch = (len + CHUNK - 1) / CHUNK;
  const uint64_t pol = l2_evict_first_policy();
  const uint8_t* gsrc = M.data + gbase;
  uint32_t issued = nch < NSLOT ? nch : NSLOT;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NSLOT; ++i) mbar_init(bar_a + 8 * i, 1);
    fence_mbarrier_init();
    for (uint32_t i = 0; i < issued; ++i) {
      const uint32_t bytes = min(static_cast<uint32_t>(CHUNK), len - i * CHUNK);
      mbar_arrive_expect_tx(bar_a + 8 * i, bytes);
      bulk_g2s(ring_a + i * CHUNK, gsrc + static_cast<uint64_t>(i) * CHUNK, bytes, bar_a + 8 * i, pol);
    }
  }
  for (int i = lane; i < NB * TILE_MAX; i += 32) acc[i] = 0.0f;
  __syncwarp();

  grid_dep_wait();

  // RMSNorm scale, when the input is rmsnorm(h): every CTA reduces h in the same order.
  float inv_rms = 1.0f;
  if (a.xs.mode == X_RMSNORM) {
    float ss = 0.0f;
    for (int k = threadIdx.x; k < a.xs.K; k += NWARPS * 32) {
      const float v = a.xs.h[k];
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) misc[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float tot = 0.0f;
      for (int w = 0; w < NWARPS; ++w) tot += misc[w];
      misc[NWARPS] = 1.0f / sqrtf(tot / static_cast<float>(a.xs.K) + a.xs.eps);
    }
    __syncthreads();
    inv_rms = misc[NWARPS];
  }
  if (a.xs.trace_x && blockIdx.x == 0) {
    for (int k = 2 * threadIdx.x; k < a.xs.K; k += 2 * NWARPS * 32) {
      const float2 v = x_pair(a.xs, 0, k, inv_rms);
      a.xs.trace_x[k] = bf16_bits(v.x);
      a.xs.trace_x[k + 1] = bf16_bits(v.y);
    }
  }

  // ---- main loop over this warp's steps ----
  bool ok = true;
  uint32_t waited = 0;
  int cur_g = -1;
  uint32_t my_desc = 0, my_off = 0, my_off1 = 0;
  for (uint32_t s = wa; s < wb; ++s) {
    const uint32_t k = (s - wa) & 31u;
    if (k == 0) {
      const uint32_t idx = s + lane;
      my_desc = idx < wb ? M.desc[idx] : 0u;
      my_off = idx < wb ? M.off[idx] : 0u;
      my_off1 = idx < wb ? M.off[idx + 1] : 0u;
    }
    const uint32_t desc = __shfl_sync(0xffffffffu, my_desc, k);
    const uint32_t o0 = static_cast<uint32_t>(static_cast<uint64_t>(__shfl_sync(0xffffffffu, my_off, k)) * 16u - gbase);
    const uint32_t o1 = static_cast<uint32_t>(static_cast<uint64_t>(__shfl_sync(0xffffffffu, my_off1, k)) * 16u - gbase);
    const uint32_t need = (o1 - 1) / CHUNK;
    while (waited <= need) {
      const bool done = mbar_wait(bar_a + 8 * (waited % NSLOT), (waited / NSLOT) & 1u);
      if (!__all_sync(0xffffffffu, done)) {
        ok = false;
        break;
      }
      ++waited;
    }
    if (!ok) break;

    const int g = static_cast<int>(desc_g(desc));
    const uint32_t cls = desc_cls(desc), e = desc_e(desc);
    if (g != cur_g) {
      __syncwarp();
#pragma unroll
      for (int c = 0; c < NB; ++c) {
        const float2 xv = x_pair(a.xs, c, g * GROUP + 2 * lane, inv_rms);
        build_prep(xp + c * XPF, xv.x, xv.y, lane);
      }
      __syncwarp();
      cur_g = g;
    }
    const uint32_t j = static_cast<uint32_t>(lane) >> cls;
    const uint32_t sigma = static_cast<uint32_t>(lane) & ((1u << cls) - 1u);
    const bool active = j < e;
    uint2 cw = make_uint2(0u, 0u);
    if (active) cw = lds_v2(ring_a + ((o0 + 8u * lane) & (RING - 1)));
    float tv[NB];
    if (cls == 0) {
      decode_lut<NB>(cw, xp_a, tv);
    } else if (cls == 1) {
      decode_direct<NB, 2>(cw, xp, sigma, tv);
#pragma unroll
      for (int c = 0; c < NB; ++c) tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 1);
    } else if (cls == 2) {
      decode_direct<NB, 4>(cw, xp, sigma, tv);
#pragma unroll
      for (int c = 0; c < NB; ++c) {
        tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 1);
        tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 2);
      }
    } else {
      decode_direct<NB, 8>(cw, xp, sigma, tv);
#pragma unroll
      for (int c = 0; c < NB; ++c) {
        tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 1);
        tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 2);
        tv[c] += __shfl_xor_sync(0xffffffffu, tv[c], 4);
      }
    }
    if (active && sigma == 0) {
      const float sc = half_bits_to_float(lds_u16(ring_a + ((o0 + rec_scale_off(cls, e) + 2u * j) & (RING - 1))));
      const uint32_t row = lds_u8(ring_a + ((o0 + rec_row_off(cls, e) + j) & (RING - 1)));
#pragma unroll
      for (int c = 0; c < NB; ++c) acc[c * TILE_MAX + row] = fmaf(sc, tv[c], acc[c * TILE_MAX + row]);
    }
    // Refill the ring with chunks whose slots are now free.
    __syncwarp();
    if (lane == 0) {
      const uint32_t lim = o1 / CHUNK + NSLOT - 1;
      while (issued < nch && issued <= lim) {
        const uint32_t slot = issued % NSLOT;
        const uint32_t bytes = min(static_cast<uint32_t>(CHUNK), len - issued * CHUNK);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar_a + 8 * slot, bytes);
        bulk_g2s(ring_a + slot * CHUNK, gsrc + static_cast<uint64_t>(issued) * CHUNK, bytes, bar_a + 8 * slot, pol);
        ++issued;
      }
    }
    __syncwarp();
  }
  if (!ok) {
    if (lane == 0) atomicExch(a.err, kErrRingTimeout);
    // Drain this warp's copies in flight (bounded) before the shared memory is released.
    for (uint32_t c = waited; c < issued; ++c)
      if (!__all_sync(0xffffffffu, mbar_wait(bar_a + 8 * (c % NSLOT), (c / NSLOT) & 1u))) break;
  }
  grid_dep_launch();

  // ---- combine: warps (fixed order), then the cluster's CTAs (fixed order) ----
  __syncthreads();
  for (uint32_t r = threadIdx.x; r < rows; r += NWARPS * 32) {
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      float v = 0.0f;
      const float* ac = reinterpret_cast<const float*>(smem + L::kAcc) + c * TILE_MAX + r;
#pragma unroll
      for (int w = 0; w < NWARPS; ++w) v += ac[w * NB * TILE_MAX];
      part[c * TILE_MAX + r] = v;
    }
  }
  cluster.sync();
  const uint32_t lo = static_cast<uint32_t>((static_cast<uint64_t>(rows) * rank) / C);
  const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(rows) * (rank + 1)) / C);
  for (uint32_t r = lo + threadIdx.x; r < hi; r += NWARPS * 32) {
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      float v = 0.0f;
      for (int q = 0; q < C; ++q) v += cluster.map_shared_rank(part, q)[c * TILE_MAX + r];
      const uint32_t row = r0 + r;
      if (M.trace_y) M.trace_y[row] = v;
      if (a.ep == EP_RESID) v += a.resid[row];
      M.y[static_cast<int64_t>(c) * M.y_ld + row] = v;
    }
  }
  cluster.sync();
}

}  // namespace vbq
