// Dequant-MMA for batches of 16..64 columns: Y = W X on the 5th-generation tensor cores.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): the packed per-group
// codes are dequantized and multiplied in one pass. With 16 or more activation
// columns the product is a real dense contraction, so this kernel rebuilds
// each (row tile, group column) of W as fp16 in shared memory and feeds it to
// tcgen05.mma. The design is this library's own, for sm_103a:
//
//  * Work: a host plan of whole (tile, column) units per CTA (plan.h,
//    whole-column mode). One CTA per SM, 8 warps.
//  * Stream: one thread copies each column's records (at most 17,408 bytes)
//    into a 3-stage shared-memory ring with cp.async.bulk; every wait is
//    bounded.
//  * Dequant: the warps decode the column's steps into A = s_g * (q - c_b),
//    rounded once to fp16, as a 256 x 64 tile, K-major with the 128-byte
//    swizzle (two 128-row halves). rows of the tile beyond its row count stay
//    zero. B is the column's 64 activations of each batch column, times a
//    per-column power of two that keeps every value inside fp16's range, as an
//    N x 64 tile in the same layout (N = batch rounded up to 16, zero rows past
//    the batch).
//  * MMA: one thread issues tcgen05.mma.cta_group::1.kind::f16 (M = 128, N,
//    K = 16, four K-steps per half) into fp32 accumulators in tensor memory,
//    then tcgen05.commit to an mbarrier. A and B are double-buffered, so the
//    warps dequantize the next column while the tensor cores run.
//  * Epilogue: tcgen05.ld of each warp's 32-lane quadrant, divided by the
//    column's power of two; a tile cut between CTAs adds its partials in split
//    order, as in the CUDA-core GEMV.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <string>

#include "internal.h"
#include "launch.h"

namespace vbq {

namespace {

constexpr int TC_WARPS = 8;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int TC_NMAX = 64;            // batch columns per launch
constexpr int TC_STAGE = 17408;        // bytes of the largest column: 64 full 8-bit steps
constexpr int TC_NST = 3;              // column stages
constexpr int TC_MAX_RUNS = 1024;      // runs of one unit (K <= 16384)
constexpr int TC_ATILE = 256 * 128;    // fp16 A tile: 256 rows x 64 K
constexpr int TC_BTILE = TC_NMAX * 128;

struct TcSmem {
  static constexpr int kA = 0;                                   // [2][256 x 128 B], 1024-aligned
  static constexpr int kB = kA + 2 * TC_ATILE;                   // [2][64 x 128 B]
  static constexpr int kStage = kB + 2 * TC_BTILE;               // [TC_NST][TC_STAGE]
  static constexpr int kDesc = kStage + TC_NST * TC_STAGE;       // unit run descriptors
  static constexpr int kOff = kDesc + TC_MAX_RUNS * 4;           // unit run offsets (16 B units, column-relative later)
  static constexpr int kCol = kOff + (TC_MAX_RUNS + 1) * 4;      // first run of each column of the unit, + end
  static constexpr int kSx = kCol + (TC_MAX_RUNS + 1) * 4;       // per batch column scale
  static constexpr int kBar = kSx + TC_NMAX * 4;                 // stage bars [3], mma bars [2]
  static constexpr int kMisc = kBar + 8 * 8;
  static constexpr int kBytes = kMisc + 64 + 1024;  // + room to align the tiles to 1024 bytes
};

struct TcArgs {
  const uint8_t* data;
  const uint32_t* run_desc;
  const uint32_t* run_off;
  const uint32_t* tile_run0;
  const UnitRec* units;   // CTA c: slots [c*umax, (c+1)*umax)
  const SliceRec* slices; // slice 0 of each unit gives its first run
  int32_t umax;
  float* partial;
  uint32_t* counters;
  const uint16_t* X;      // bf16 [B][K]
  const float* sx;        // [B] powers of two
  float* Y;               // [B][N]
  int32_t B, Npad, K, N;
  int* err;
};

// A and B tiles: element (row, k) of an 8-row-atom, 128-byte-swizzled, K-major tile.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// K order inside one 64-wide group column (both A and B use it): position
// 32*blk + 2*s + h holds code 32*blk + s + 16*h (s < 16, h < 2). A 32-bit code
// plane then yields the pair (s, s + 16) with one shift and one mask, and an
// 8-bit lane slice with one byte permute. The product does not depend on the
// order of K.

// Dequantization to fp16 without conversions: 0x6400 | q is the fp16 value
// 1024 + q (q < 1024). With c = (2^b - 1)/2 = m0 + 1/2, (1024 + q) - (1024 + m0)
// = q - m0 exactly, and fma(q - m0, s, -s/2) = s * (q - c) rounded once
// (s/2 is exact in fp16).
__device__ __forceinline__ uint32_t deq_pair(uint32_t h1024q, __half2 base, __half2 sc, __half2 nhs) {
  const __half2 v = __hfma2(__hsub2(*reinterpret_cast<const __half2*>(&h1024q), base), sc, nhs);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void put16(uint8_t* sm, uint32_t a_base, uint32_t row, uint32_t chunk, uint4 v) {
  *reinterpret_cast<uint4*>(sm + a_base + (row >> 7) * (TC_ATILE / 2) + sw128(row & 127u, chunk)) = v;
}

// Decodes one step of class CLS (e entries) at shared offset rb into A.
template <int CLS>
__device__ __forceinline__ void tc_step_cls(uint8_t* sm, uint32_t rb, uint32_t e, uint32_t a_base, int lane) {
  constexpr uint32_t B = 1u << CLS;
  const uint32_t j = static_cast<uint32_t>(lane) >> CLS;
  const uint32_t sg = static_cast<uint32_t>(lane) & (B - 1u);
  const bool active = j < e;
  const uint2 cw = *reinterpret_cast<const uint2*>(sm + rb + 8u * lane);  // in the ring or its spill zone
  const uint16_t sb = *reinterpret_cast<const uint16_t*>(sm + rb + rec_scale_off(CLS, e) + 2u * j);
  const uint32_t row = sm[rb + rec_row_off(CLS, e) + j];
  const __half2 sc = __half2half2(__ushort_as_half(sb));
  const __half2 nhs = __hmul2(sc, __float2half2_rn(-0.5f));
  const __half2 base = __float2half2_rn(static_cast<float>(1024u + (1u << (B - 1u)) - 1u));
  if constexpr (CLS == 3) {
    // Lane sg holds codes 8 sg .. 8 sg + 7; it writes chunk sg, which holds codes
    // 32 blk + 4 t0 + i and those + 16 (blk = sg / 4, t0 = sg % 4, i < 4).
    const int src = (lane & ~7) | static_cast<int>(4u * (sg >> 2) + ((sg & 3u) >> 1));
    const uint32_t ax = __shfl_sync(0xffffffffu, cw.x, src), ay = __shfl_sync(0xffffffffu, cw.y, src);
    const uint32_t bx = __shfl_sync(0xffffffffu, cw.x, src + 2), by = __shfl_sync(0xffffffffu, cw.y, src + 2);
    const uint32_t a = (sg & 1u) ? ay : ax, b = (sg & 1u) ? by : bx;
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pr = __byte_perm(a, b, static_cast<uint32_t>(i | (i << 4) | ((4 + i) << 8) | ((4 + i) << 12)));
      o[i] = deq_pair((pr & 0x00FF00FFu) | 0x64006400u, base, sc, nhs);
    }
    if (active) put16(sm, a_base, row, sg, make_uint4(o[0], o[1], o[2], o[3]));
  } else {
    // Gather the entry's B planes; lane sg writes chunks sg * 8 / B .. + 8 / B - 1.
    // Plane word w is kept as the 64-bit value w << 8 (hi:lo), so that one
    // funnel shift right by s + 8 - p puts its bits s and s + 16 at bits p and
    // 16 + p.
    uint32_t lo[2][B], hi[2][B];
#pragma unroll
    for (uint32_t p = 0; p < B; ++p) {
      const int src = (lane & ~static_cast<int>(B - 1u)) | static_cast<int>(p);
      const uint32_t x = __shfl_sync(0xffffffffu, cw.x, src), y = __shfl_sync(0xffffffffu, cw.y, src);
      lo[0][p] = x << 8;
      hi[0][p] = x >> 24;
      lo[1][p] = y << 8;
      hi[1][p] = y >> 24;
    }
    if (!active) return;
#pragma unroll
    for (uint32_t cc = 0; cc < 8u / B; ++cc) {
      const uint32_t c = sg * (8u / B) + cc;
      const uint32_t wsel = c >> 2, s0 = 4u * (c & 3u);
      uint32_t o[4];
#pragma unroll
      for (uint32_t t = 0; t < 4; ++t) {
        uint32_t q = 0x64006400u;
#pragma unroll
        for (uint32_t p = 0; p < B; ++p)
          q |= __funnelshift_r(wsel ? lo[1][p] : lo[0][p], wsel ? hi[1][p] : hi[0][p], s0 + t + 8u - p) &
               (0x00010001u << p);
        o[t] = deq_pair(q, base, sc, nhs);
      }
      put16(sm, a_base, row, c, make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
}

__device__ __forceinline__ void tc_step(uint8_t* sm, uint32_t rb, uint32_t cls, uint32_t e, uint32_t a_base,
                                        int lane) {
  switch (cls) {
    case 0: tc_step_cls<0>(sm, rb, e, a_base, lane); break;
    case 1: tc_step_cls<1>(sm, rb, e, a_base, lane); break;
    case 2: tc_step_cls<2>(sm, rb, e, a_base, lane); break;
    default: tc_step_cls<3>(sm, rb, e, a_base, lane); break;
  }
}

__global__ void __launch_bounds__(TC_THREADS, 1) vbq_gemm_tc_kernel(const __grid_constant__ TcArgs a) {
  using L = TcSmem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Every region sits at its offset from the first 1024-byte boundary of the dynamic shared memory.
  const uint32_t sraw = smem_u32(vbq_smem);
  const uint32_t pad = ((sraw + 1023u) & ~1023u) - sraw;
  uint8_t* const sm = vbq_smem + pad;
  const uint32_t sbase = sraw + pad;
  uint32_t* descs = reinterpret_cast<uint32_t*>(sm + L::kDesc);
  uint32_t* offs = reinterpret_cast<uint32_t*>(sm + L::kOff);
  uint32_t* cols = reinterpret_cast<uint32_t*>(sm + L::kCol);
  float* sxs = reinterpret_cast<float*>(sm + L::kSx);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  const uint32_t bar_stage = sbase + L::kBar;       // 3 stage barriers
  const uint32_t bar_mma = sbase + L::kBar + 24;    // 2 MMA barriers
  const int N = a.Npad;

  // Units of this CTA.
  int nu = 0;
  while (nu < a.umax && a.units[static_cast<size_t>(blockIdx.x) * a.umax + nu].nsplit > 0) ++nu;

  if (tid == 0) {
    for (int i = 0; i < TC_NST; ++i) mbar_init(bar_stage + 8 * i, 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar_mma + 8 * i, 1);
    fence_mbarrier_init();
  }
  for (int i = tid; i < TC_NMAX; i += TC_THREADS) sxs[i] = i < a.B ? a.sx[i] : 0.0f;
  if (warp == 0) {
    tmem_alloc(sbase + L::kMisc, 2 * TC_NMAX);  // 128 columns: two 128-lane halves of N <= 64 columns
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  bool ok = true;
  const uint64_t pol = l2_evict_first_policy();
  const uint32_t idesc = tc_idesc_f16(128, static_cast<uint32_t>(N));

  uint32_t gcol = 0;      // columns processed by this CTA so far (all units)
  uint32_t issued = 0;    // columns of the current unit whose copy has been issued (thread 0)
  uint32_t issued_g = 0;  // columns of all units whose copy has been issued (thread 0)
  uint32_t mma_g = 0;     // columns whose MMAs have been issued and committed (thread 0)

  for (int u = 0; u < nu && ok; ++u) {
    const size_t slot = static_cast<size_t>(blockIdx.x) * a.umax + u;
    const UnitRec ur = a.units[slot];
    const SliceRec s0 = a.slices[slot * SLICES];
    const SliceRec sl = a.slices[slot * SLICES + SLICES - 1];
    const uint32_t run_a = s0.run0, run_b = sl.run1;  // whole runs (k = 0 at both ends)
    const uint32_t nruns = run_b - run_a;
    // Unit metadata into shared memory.
    for (uint32_t i = tid; i < nruns; i += TC_THREADS) descs[i] = a.run_desc[run_a + i];
    for (uint32_t i = tid; i <= nruns; i += TC_THREADS) offs[i] = a.run_off[run_a + i];
    __syncthreads();
    // Column starts within the unit.
    if (tid == 0) {
      uint32_t nc = 0;
      for (uint32_t i = 0; i < nruns; ++i)
        if (i == 0 || run_g(descs[i]) != run_g(descs[i - 1])) cols[nc++] = i;
      cols[nc] = nruns;
      misc[1] = nc;
    }
    // Zero the rows past the tile in both A buffers (the MMA of a half with no rows is skipped).
    const uint32_t rows = ur.rows;
    for (uint32_t i = tid; i < (256u - rows) * 8u; i += TC_THREADS) {
      const uint32_t row = rows + i / 8u, ch = i % 8u;
      for (int p = 0; p < 2; ++p)
        *reinterpret_cast<uint4*>(sm + L::kA + p * TC_ATILE + (row >> 7) * (TC_ATILE / 2) + sw128(row & 127u, ch)) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    const uint32_t ncols = misc[1];
    const bool two_halves = rows > 128u;

    // Copies of this unit's first columns (the stages are free: the previous unit is done).
    const uint32_t gcol0 = gcol;
    auto issue_col = [&](uint32_t c) {  // thread 0 only; column c of this unit
      const uint32_t st = (gcol0 + c) % TC_NST;
      fence_proxy_async_smem();
      const uint32_t o0 = offs[cols[c]], o1 = offs[cols[c + 1]];
      const uint32_t bytes = (o1 - o0) * 16u;
      mbar_arrive_expect_tx(bar_stage + 8 * st, bytes);
      bulk_g2s(sbase + L::kStage + st * TC_STAGE, a.data + static_cast<uint64_t>(o0) * 16u, bytes, bar_stage + 8 * st,
               pol);
      ++issued_g;
    };
    if (tid == 0) {
      for (uint32_t c = 0; c < ncols && c < TC_NST; ++c) issue_col(c);
      issued = ncols < TC_NST ? ncols : TC_NST;
    }

    for (uint32_t c = 0; c < ncols; ++c, ++gcol) {
      const uint32_t st = gcol % TC_NST;
      const uint32_t buf = gcol & 1u;
      // The MMAs that last read this A/B buffer (two columns ago) must be done.
      if (gcol >= 2) {
        const bool done = mbar_wait(bar_mma + 8 * buf, ((gcol >> 1) - 1u) & 1u);
        if (!__syncthreads_and(done)) {
          ok = false;
          break;
        }
      }
      // This column's records.
      const bool landed = mbar_wait(bar_stage + 8 * st, (gcol / TC_NST) & 1u);
      if (!__syncthreads_and(landed)) {
        ok = false;
        break;
      }
      const uint32_t a_base = L::kA + buf * TC_ATILE;
      const uint32_t rec0 = L::kStage + st * TC_STAGE;
      const uint32_t o0 = offs[cols[c]];
      const uint32_t g = run_g(descs[cols[c]]);
      // Dequantize: warps take the column's steps in turn.
      uint32_t sidx = 0;
      for (uint32_t r = cols[c]; r < cols[c + 1]; ++r) {
        const uint32_t d = descs[r];
        const uint32_t cls = run_cls(d), n = run_n(d), eps = entries_per_step(cls);
        const uint32_t nst = (n + eps - 1u) / eps;
        const uint32_t rbase = rec0 + (offs[r] - o0) * 16u;
        for (uint32_t k = 0; k < nst; ++k, ++sidx) {
          if (static_cast<int>(sidx % TC_WARPS) != warp) continue;
          tc_step(sm, rbase + k * full_step_bytes(cls), cls, min(eps, n - k * eps), a_base, lane);
        }
      }
      // B: the column's activations, scaled into fp16 range, rows past the batch zero.
      const uint32_t b_base = L::kB + buf * TC_BTILE;
      for (int i = tid; i < N * 8; i += TC_THREADS) {
        const int bc = i >> 3, ch = i & 7;
        uint4 pk = make_uint4(0u, 0u, 0u, 0u);
        if (bc < a.B) {
          // Chunk ch holds codes 32 blk + s0 + t and those + 16 (t < 4), in pairs.
          const uint16_t* xr = a.X + static_cast<int64_t>(bc) * a.K + g * GROUP + 32 * (ch >> 2) + 4 * (ch & 3);
          const uint2 lo4 = *reinterpret_cast<const uint2*>(xr), hi4 = *reinterpret_cast<const uint2*>(xr + 16);
          const float s = sxs[bc];
          const float xa[4] = {bf16_lo(lo4.x), bf16_hi(lo4.x), bf16_lo(lo4.y), bf16_hi(lo4.y)};
          const float xb[4] = {bf16_lo(hi4.x), bf16_hi(hi4.x), bf16_lo(hi4.y), bf16_hi(hi4.y)};
          uint32_t o[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            o[t] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(xa[t] * s))) |
                   (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(xb[t] * s))) << 16);
          pk = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4*>(sm + b_base + sw128(static_cast<uint32_t>(bc), static_cast<uint32_t>(ch))) = pk;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        for (uint32_t h = 0; h < (two_halves ? 2u : 1u); ++h) {
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk) {
            const uint64_t ad = tc_desc_sw128(sbase + a_base + h * (TC_ATILE / 2) + kk * 32u, 1024u);
            const uint64_t bd = tc_desc_sw128(sbase + b_base + kk * 32u, 1024u);
            tc_mma_f16(tmem + h * static_cast<uint32_t>(N), ad, bd, idesc, c > 0 || kk > 0);
          }
        }
        tc_commit(bar_mma + 8 * buf);
        ++mma_g;
        // The stage of this column is free again: bring in column c + TC_NST.
        if (issued < ncols) {
          issue_col(issued);
          ++issued;
        }
      }
    }
    if (!ok) break;

    // ---- epilogue: all MMAs of the unit are done when the last commit has arrived ----
    {
      const uint32_t last = gcol - 1u;
      const bool done = mbar_wait(bar_mma + 8 * (last & 1u), (last >> 1) & 1u);
      if (!__syncthreads_and(done)) {
        ok = false;
        break;
      }
    }
    tc_fence_after();
    const uint32_t quad = static_cast<uint32_t>(warp & 3), half = static_cast<uint32_t>(warp >> 2);
    const uint32_t r = half * 128u + quad * 32u + static_cast<uint32_t>(lane);
    const bool has_row = r < rows && (half == 0 || two_halves);
    float* part = ur.nsplit > 1 ? a.partial + static_cast<size_t>(ur.pbase) * a.B : nullptr;
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + ((quad * 32u) << 16) + half * static_cast<uint32_t>(N) + static_cast<uint32_t>(c0), v);
      tmem_ld_wait();
      if (has_row && (half == 0 || two_halves)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int bc = c0 + i;
          if (bc < a.B) {
            const float y = __uint_as_float(v[i]) / sxs[bc];
            if (part) part[(ur.split * a.B + bc) * rows + r] = y;
            else a.Y[static_cast<int64_t>(bc) * a.N + ur.r0 + r] = y;
          }
        }
      }
    }
    tc_fence_before();
    if (ur.nsplit > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) misc[2] = (atomicAdd(a.counters + ur.cnt, 1u) == ur.nsplit - 1u) ? 1u : 0u;
      __syncthreads();
      if (misc[2]) {
        __threadfence();
        for (uint32_t i = tid; i < rows * static_cast<uint32_t>(a.B); i += TC_THREADS) {
          const uint32_t bc = i / rows, rr = i % rows;
          float y = 0.0f;
          for (uint32_t s = 0; s < ur.nsplit; ++s) y += __ldcg(part + (s * a.B + bc) * rows + rr);
          a.Y[static_cast<int64_t>(bc) * a.N + ur.r0 + rr] = y;
        }
        if (tid == 0) a.counters[ur.cnt] = 0u;
      }
    }
    __syncthreads();  // the accumulators are read before the next unit overwrites them
    tc_fence_after();
  }

  if (!ok && tid == 0) {
    atomicExch(a.err, kErrMmaTimeout);
    // Wait (bounded) for the copies and MMAs still in flight before the memory goes away.
    for (uint32_t c = gcol; c < issued_g; ++c) (void)mbar_wait(bar_stage + 8 * (c % TC_NST), (c / TC_NST) & 1u);
    if (mma_g > 0) {
      const uint32_t last = mma_g - 1u;
      (void)mbar_wait(bar_mma + 8 * (last & 1u), (last >> 1) & 1u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * TC_NMAX);
}

// x scale per batch column: a power of two s with max|x| * s in [2^13, 2^14).
__global__ void vbq_xscale_kernel(const uint16_t* __restrict__ X, int32_t K, float* __restrict__ sx) {
  __shared__ float red[32];
  const uint16_t* x = X + static_cast<int64_t>(blockIdx.x) * K;
  float m = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[k]) << 16)));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    m = fmaxf(m, red[0]);
    int e = 0;
    (void)frexpf(m, &e);  // m = f * 2^e, f in [0.5, 1)
    int p = m > 0.0f ? 14 - e : 0;
    p = p > 100 ? 100 : (p < -100 ? -100 : p);
    sx[blockIdx.x] = ldexpf(1.0f, p);
  }
}

}  // namespace

// Per-matrix tensor-core state, made on the first batch of 16 or more columns.
struct TcState {
  DevicePlan plan;
  float* sx = nullptr;
  bool ok = false;
};

static std::mutex g_tc_mu;
static std::map<const vbq_matrix*, TcState> g_tc;

void tc_forget(const vbq_matrix* m) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  auto it = g_tc.find(m);
  if (it == g_tc.end()) return;
  free_plan(&it->second.plan);
  if (it->second.sx) cudaFree(it->second.sx);
  g_tc.erase(it);
}

bool tc_eligible(const vbq_matrix* m) {
  if (m->tc_max_scale > 512.0f) return false;  // s * 127.5 must stay inside fp16
  if (m->K % 8 != 0) return false;
  if (m->max_col_bytes > TC_STAGE) return false;  // a column's records must fit one stage
  // every unit's runs must fit the shared-memory run table
  const int64_t runs_per_tile_max = 4 * static_cast<int64_t>(m->G);
  return runs_per_tile_max <= TC_MAX_RUNS;
}

static vbq_status tc_state(const vbq_matrix* m, TcState** out) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  TcState& s = g_tc[m];
  if (!s.ok) {
    Plan pl = make_plan({seg_tables(m)}, plan_ctas(static_cast<uint64_t>(m->data_bytes), gpu_info().sms),
                        MAX_UNITS_PER_CTA, true);
    cudaError_t e = upload_plan(pl, TC_NMAX, {m->data}, nullptr, &s.plan);
    if (e != cudaSuccess) return cuda_fail(e, "vbq_gemm_smallbatch: tensor-core plan");
    e = cudaMalloc(&s.sx, TC_NMAX * sizeof(float));
    if (e != cudaSuccess) {
      free_plan(&s.plan);
      return cuda_fail(e, "vbq_gemm_smallbatch: scale scratch");
    }
    cudaFuncSetAttribute(vbq_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kBytes);
    s.ok = true;
  }
  *out = &s;
  return VBQ_OK;
}

vbq_status launch_gemm_tc(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st) {
  if (B < 16 || B > TC_NMAX) return fail(VBQ_ERR_INVALID_ARG, "tensor-core path: batch out of range");
  TcState* s = nullptr;
  vbq_status r = tc_state(m, &s);
  if (r != VBQ_OK) return r;
  int* err = device_check_word();
  if (!err) return fail(VBQ_ERR_CUDA, "device check word");
  note_launches(1);
  vbq_xscale_kernel<<<B, 256, 0, st>>>(X, static_cast<int32_t>(m->K), s->sx);
  VBQ_CUDA_TRY(cudaGetLastError());
  if (s->plan.n_ctas <= 0) return VBQ_OK;
  TcArgs a{};
  a.data = m->data;
  a.run_desc = m->run_desc;
  a.run_off = m->run_off;
  a.tile_run0 = m->tile_run0;
  a.units = s->plan.units;
  a.slices = s->plan.slices;
  a.umax = s->plan.umax;
  a.partial = s->plan.partial;
  a.counters = s->plan.counters;
  a.X = X;
  a.sx = s->sx;
  a.Y = Y;
  a.B = B;
  a.Npad = (B + 15) & ~15;
  a.K = static_cast<int32_t>(m->K);
  a.N = static_cast<int32_t>(m->N);
  a.err = err;
  note_launches(1);
  vbq_gemm_tc_kernel<<<s->plan.n_ctas, TC_THREADS, TcSmem::kBytes, st>>>(a);
  VBQ_CUDA_TRY(cudaGetLastError());
  return VBQ_OK;
}

}  // namespace vbq
