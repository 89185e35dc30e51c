// Fused dequantize-and-multiply for the packed VBQ layout (layout.h), batch 1,
// on the CUDA cores: the building blocks shared by the single-GEMV kernel and
// the persistent decode-step kernel.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): decode is memory-bound,
// and the packed per-group codes are dequantized inside the multiply. The
// abstract's kernels ran on Apple silicon; these are this library's own design
// for sm_103a. Measured rates on this GPU, in warp instructions per clock per
// SM: shuffle 1, dp2a/dp4a 2 (own pipe), LOP3/SHF/PRMT 2, FFMA 4. A 1-bit step
// (13 shuffles) is bound by the shared-memory/shuffle pipe.
//
//  * Fixed point. Every partial sum of a row is at most L1 * max|x|, with L1
//    the largest row sum of |w| (known when packing). With F = 30 - ceil(log2
//    of that bound), each entry's contribution is rounded to an integer in
//    units of 2^-F and added with integer atomics: into 32-bit row
//    accumulators in shared memory (one per CTA), then into 64-bit sums in
//    global memory. Integer adds do not depend on their order, so results are
//    deterministic, and the rounding costs about 2^-31 of the bound per entry.
//  * Staging. Each CTA stages the group columns its range touches (at most
//    CCAP): x * 2^F in "lookup order" (fp32 pairs for building 1-bit tables two
//    at a time), a 16-bit fixed-point copy X = rint(x * 2^s_g) with |X| < 2^14,
//    and per column sum(X) and 2^(F - s_g - 1).
//  * Streaming. Each warp streams its byte range through a private ring of NS
//    4 KB shared-memory slots with cp.async.bulk copies completed on mbarriers
//    (all waits bounded). The first SPILL bytes of each copy into slot 0 are
//    also written past the ring's end, so a record that crosses the end is
//    read without wrapping.
//  * 1-bit runs: lane l holds T_k[l] = sum_{i<5} (bit_i(l) - 1/2) x'_{5k+i} for
//    k = 0..12; a 64-bit code word is 13 x (shift, shuffle, add), giving
//    sum_m (q_m - 1/2) x'_m as the group's dot product.
//  * 2-, 4- and 8-bit runs: (word >> (b*i)) & mask puts four codes in the four
//    bytes of a register (layout.h) and dp2a multiplies them with two int16
//    pairs of X; the sums are exact integers. The lanes of an entry are added
//    with shuffles, and sum (q - c_b) X = sum q X - c_b sum X.
#pragma once

#include "layout.h"
#include "plan.h"
#include "ptx.cuh"

namespace vbq {

#ifndef VBQ_LOG_CH
#define VBQ_LOG_CH 12
#endif
constexpr int LOG_CH = VBQ_LOG_CH;
constexpr int CH = 1 << LOG_CH;      // bytes per bulk copy and per ring slot
constexpr int NS_MAX = 16;           // ring slots per warp at most
constexpr int SPILL = 2176;          // bytes past the ring's end (>= header + the largest record)
constexpr int XL_FLOATS = 72;        // per column: 7 x 5 float2 in lookup order, padded to 16 bytes
constexpr int NLUT = 13;             // 5-bit tables per group (the last covers 4 codes)
constexpr int XCAP = 16384;          // largest K of the batch-1 kernels
constexpr uint32_t kNoRefill = 0xFFFFFFFFu;

// Build-time tuning: ring slots per warp, and steps decoded together (1-bit
// runs, and 2/4/8-bit runs).
#ifndef VBQ_NS
#define VBQ_NS 2
#endif
#ifndef VBQ_U1
#define VBQ_U1 2
#endif
#ifndef VBQ_UDP
#define VBQ_UDP 1
#endif
constexpr int kRingSlots = VBQ_NS;
constexpr int kU1 = VBQ_U1;
constexpr int kUdp = VBQ_UDP;
static_assert(kRingSlots >= 2 && kRingSlots <= NS_MAX, "ring slots");
static_assert(CH >= 512 && (kRingSlots - 1) * CH >= 1024, "a few steps must fit ahead of the consumer");
static_assert(SPILL % 16 == 0 && SPILL <= CH && SPILL >= HEADER_BYTES + full_step_bytes(3),
              "a record that crosses the ring's end must fit in the mirrored bytes");
// A warp waits for the bytes of U steps past its position; they must fit in
// the slots other than the one being read.
static_assert(kU1 * full_step_bytes(0) <= (kRingSlots - 1) * CH && kUdp * full_step_bytes(3) <= (kRingSlots - 1) * CH,
              "steps decoded together must fit in the ring");

struct ColInfo {
  int32_t sum_x;  // sum of the column's 64 fixed-point values
  float u;        // 2^(F - s_g - 1): one unit of 2 * sum (q - c) X, in units of 2^-F
};

// Shared-memory layout of the batch-1 kernels with NS ring slots per warp.
struct SmemLayout {
  uint32_t ring_stride, ring, acc, xl, X, col, bar, misc, total;
};
__host__ __device__ inline constexpr SmemLayout smem_layout(int ns) {
  SmemLayout L{};
  L.ring_stride = static_cast<uint32_t>(ns) * CH + SPILL;
  L.ring = 0;
  L.acc = L.ring + KW * L.ring_stride;
  L.xl = L.acc + SLOTS_MAX * SROWS * 4;
  L.X = L.xl + CCAP * XL_FLOATS * 4;
  L.col = L.X + CCAP * 128;
  L.bar = L.col + CCAP * 8;
  L.misc = L.bar + KW * NS_MAX * 8;
  L.total = L.misc + 512;
  return L;
}

extern __shared__ __align__(1024) uint8_t vbq_smem[];

template <typename T>
__device__ __forceinline__ T lds(uint32_t off) {
  return *reinterpret_cast<const T*>(vbq_smem + off);
}
template <typename T>
__device__ __forceinline__ void sts(uint32_t off, T v) {
  *reinterpret_cast<T*>(vbq_smem + off) = v;
}

__device__ __forceinline__ void red_shared_add_s32(uint32_t addr, int v) {
  asm volatile("red.shared.add.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---- fixed point -------------------------------------------------------------

// F = 30 - e with max_row_l1 * max|x| < 2^e: every partial sum of a row, in
// units of 2^-F, stays below 2^30 in magnitude.
__device__ __forceinline__ int fixed_exponent(float max_row_l1, float max_abs_x) {
  if (!(max_abs_x > 0.0f) || !(max_row_l1 > 0.0f)) return 0;
  int el, ex;
  frexpf(max_row_l1, &el);
  frexpf(max_abs_x, &ex);
  return 30 - (el + ex);
}

// ---- staging of x ------------------------------------------------------------

// 2^e as a float for -126 <= e <= 127 (exact).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }
// v * 2^e, exact unless the result leaves the float range (two steps when 2^e does).
__device__ __forceinline__ float mul_pow2(float v, int e) {
  if (e >= -126 && e <= 127) return v * pow2f(e);
  return scalbnf(v, e);
}
// The e with m < 2^e, for m > 0 (as frexpf gives it).
__device__ __forceinline__ int exp_above(float m) {
  const uint32_t b = __float_as_uint(m);
  if ((b >> 23) != 0u) return static_cast<int>(b >> 23) - 126;
  int e;
  frexpf(m, &e);  // subnormal
  return e;
}

// Stores NC columns into staging slots j0 + q * jstep (q < NC, only those
// below ncols): lane l gives x_{2l} and x_{2l+1} of each (bf16 values held in
// floats). Whole warp; the columns' reductions are interleaved. F is the
// fixed-point exponent.
template <int NC>
__device__ __forceinline__ void put_columns(const SmemLayout& L, uint32_t j0, uint32_t jstep, uint32_t ncols,
                                           const float (&x0)[NC], const float (&x1)[NC], int F, int lane) {
  float m[NC];
#pragma unroll
  for (int q = 0; q < NC; ++q) m[q] = fmaxf(fabsf(x0[q]), fabsf(x1[q]));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1)
#pragma unroll
    for (int q = 0; q < NC; ++q) m[q] = fmaxf(m[q], __shfl_xor_sync(0xffffffffu, m[q], d));
  int s[NC], sx[NC], X0[NC], X1[NC];
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    s[q] = m[q] > 0.0f ? 14 - exp_above(m[q]) : 0;  // |x| * 2^s < 2^14
    X0[q] = __float2int_rn(mul_pow2(x0[q], s[q]));
    X1[q] = __float2int_rn(mul_pow2(x1[q], s[q]));
    sx[q] = X0[q] + X1[q];
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1)
#pragma unroll
    for (int q = 0; q < NC; ++q) sx[q] += __shfl_xor_sync(0xffffffffu, sx[q], d);
#pragma unroll
  for (int q = 0; q < NC; ++q) {
    const uint32_t j = j0 + q * jstep;
    if (j >= ncols) continue;
    sts<uint32_t>(L.X + j * 128 + 4 * lane, (static_cast<uint32_t>(X0[q]) & 0xFFFFu) | (static_cast<uint32_t>(X1[q]) << 16));
    // Lookup order: float2 (x'_{10p+i}, x'_{10p+5+i}) at pair p*5 + i, p = 0..6, i = 0..4, x' = x * 2^F.
    const uint32_t xb = L.xl + j * XL_FLOATS * 4;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = 2 * lane + h;
      const int p = jj / 10, w = jj - 10 * p;
      const int idx = (p * 5 + (w % 5)) * 2 + w / 5;
      sts<float>(xb + idx * 4, mul_pow2(h ? x1[q] : x0[q], F));
    }
    // x_64 .. x_69 do not exist: zero their slots (indices 68 and 61, 63, 65, 67, 69).
    if (lane < 6) sts<float>(xb + (lane == 0 ? 68 : 59 + 2 * lane) * 4, 0.0f);
    if (lane == 0) {
      ColInfo ci;
      ci.sum_x = sx[q];
      ci.u = mul_pow2(1.0f, F - s[q] - 1);
      sts<ColInfo>(L.col + j * 8, ci);
    }
  }
}

// Stages the warp's columns (slots warp, warp + KW, ...) from values given by get(j, &x0, &x1).
template <typename Get>
__device__ __forceinline__ void stage_columns(const SmemLayout& L, uint32_t ncols, int F, int lane, int warp, Get get) {
  constexpr int CPW = (CCAP + KW - 1) / KW;
  if (static_cast<uint32_t>(warp) >= ncols) return;
  if (ncols <= static_cast<uint32_t>(KW)) {  // one column for this warp
    float a[1], b[1];
    get(static_cast<uint32_t>(warp), &a[0], &b[0]);
    put_columns<1>(L, warp, KW, ncols, a, b, F, lane);
    return;
  }
  float a[CPW], b[CPW];
#pragma unroll
  for (int q = 0; q < CPW; ++q) {
    const uint32_t j = warp + q * KW;
    a[q] = b[q] = 0.0f;
    if (j < ncols) get(j, &a[q], &b[q]);
  }
  put_columns<CPW>(L, warp, KW, ncols, a, b, F, lane);
}

// ---- per-warp stream ---------------------------------------------------------

// Per-warp stream of packed bytes: ring, chunks issued and landed, and the
// producer's place in the warp's piece list. Lane 0 issues the copies; the
// bookkeeping is warp-uniform.
struct WarpStream {
  uint32_t ring;       // shared offset of the ring
  uint32_t ring_a;     // shared address of the ring
  uint32_t bar;        // shared address of the first slot's mbarrier
  uint32_t rbytes;     // ring bytes (ns * CH)
  uint32_t ns;         // slots
  uint32_t L;          // stream bytes
  uint32_t nch;        // chunks
  uint32_t issued, landed;
  uint32_t islot;      // slot of chunk `issued`
  uint32_t lslot, lphase;  // slot and phase parity of chunk `landed`
  uint32_t avail;      // bytes known to have landed
  uint32_t refill_at;  // stream offset at which the next chunk may be issued
  const uint64_t* pieces;
  uint32_t npieces;
  uint32_t pi;         // producer: piece being copied
  uint32_t ppos;       // producer: bytes of it already copied
  uint64_t pcur, pnext;  // lane i: pieces (pbase + i) and (pbase + 32 + i)
  uint32_t pbase;
  uint64_t pol;
  bool ok;

  __device__ __forceinline__ void init(uint32_t ring_off, uint32_t nslots, uint32_t bar_addr, const uint64_t* list,
                                       uint32_t n, uint32_t bytes, int lane) {
    ring = ring_off;
    ring_a = smem_u32(vbq_smem) + ring_off;
    bar = bar_addr;
    ns = nslots;
    rbytes = nslots * CH;
    L = bytes;
    nch = (bytes + CH - 1) >> LOG_CH;
    issued = landed = avail = 0;
    islot = lslot = lphase = 0;
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
      for (uint32_t i = 0; i < nslots; ++i) mbar_init(bar + 8 * i, 1);
      fence_mbarrier_init();
    }
    __syncwarp();
  }

  __device__ __forceinline__ void issue_next(int lane) {
    const uint32_t slot = islot;
    const uint32_t bytes = min(static_cast<uint32_t>(CH), L - issued * CH);
    const uint32_t spill = (slot == 0 && issued > 0) ? min(static_cast<uint32_t>(SPILL), bytes) : 0u;
    const uint32_t b = bar + 8 * slot;
    if (lane == 0) mbar_arrive_expect_tx(b, bytes + spill);
    uint32_t done = 0;
    while (done < bytes && pi < npieces) {
      if (pi - pbase >= 32u) {
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
        if (done < spill) bulk_g2s(ring_a + rbytes + done, src, min(take, spill - done), b, pol);
      }
      done += take;
      ppos += take;
      if (ppos == plen) {
        ++pi;
        ppos = 0;
      }
    }
    ++issued;
    islot = islot + 1 == ns ? 0u : islot + 1;
    refill_at = issued < nch ? (issued + 1 - ns) * CH : kNoRefill;
  }

  __device__ __forceinline__ void start(int lane) {
    while (issued < nch && issued < ns) issue_next(lane);
  }

  // Waits until the bytes below `upto` have landed; sets ok = false on a timeout.
  __device__ __forceinline__ void wait_for(uint32_t upto) {
    while (avail < upto) {
      const bool done = mbar_wait(bar + 8 * lslot, lphase);
      if (!__all_sync(0xffffffffu, done)) {
        ok = false;
        return;
      }
      ++landed;
      if (++lslot == ns) {
        lslot = 0;
        lphase ^= 1u;
      }
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
    while (landed < issued) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar + 8 * lslot, lphase))) break;
      ++landed;
      if (++lslot == ns) {
        lslot = 0;
        lphase ^= 1u;
      }
    }
  }
};

// ---- decode of one step ------------------------------------------------------

// sum_m (q_m - 1/2) x'_m of a 64-bit code word against the lookup tables.
__device__ __forceinline__ float decode_plane(uint2 cw, const float (&lut)[NLUT]) {
  const uint32_t w0 = cw.x, w1 = cw.y;
  const uint32_t f[NLUT] = {w0,       w0 >> 5,  w0 >> 10, w0 >> 15, w0 >> 20, w0 >> 25, __funnelshift_r(w0, w1, 30),
                            w1 >> 3,  w1 >> 8,  w1 >> 13, w1 >> 18, w1 >> 23, w1 >> 28};
  float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < NLUT; ++k) a[k & 3] += __shfl_sync(0xffffffffu, lut[k], static_cast<int>(f[k]));
  return (a[0] + a[1]) + (a[2] + a[3]);
}

// sum q X over the lane's 2-, 4- or 8-bit entry (exact int32): its 2b code
// words w against the column's 32 X pairs, in four independent sums.
template <int CLS>
__device__ __forceinline__ int decode_dp(const uint32_t (&w)[16], const uint32_t (&xp)[32]) {
  constexpr int NW = 2 << CLS;
  int s[4] = {0, 0, 0, 0};
#pragma unroll
  for (int k = 0; k < NW; ++k) {
    if constexpr (CLS == 1) {  // word k: codes 16k .. 16k+15
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t by = (w[k] >> (2 * i)) & 0x03030303u;
        s[i & 3] = dp2a_lo(xp[8 * k + 2 * i], by, s[i & 3]);
        s[i & 3] = dp2a_hi(xp[8 * k + 2 * i + 1], by, s[i & 3]);
      }
    } else if constexpr (CLS == 2) {  // word k: codes 8k .. 8k+7
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t by = (w[k] >> (4 * i)) & 0x0F0F0F0Fu;
        s[(2 * k + i) & 3] = dp2a_lo(xp[4 * k + 2 * i], by, s[(2 * k + i) & 3]);
        s[(2 * k + i) & 3] = dp2a_hi(xp[4 * k + 2 * i + 1], by, s[(2 * k + i) & 3]);
      }
    } else {  // word k: codes 4k .. 4k+3
      s[k & 3] = dp2a_lo(xp[2 * k], w[k], s[k & 3]);
      s[k & 3] = dp2a_hi(xp[2 * k + 1], w[k], s[k & 3]);
    }
  }
  return (s[0] + s[1]) + (s[2] + s[3]);
}

// Per-warp consumer state.
struct Worker {
  uint32_t o;        // stream offset of the next byte to consume
  uint32_t opos;     // o modulo the ring size
  int lut_col;       // staging slot whose lookup tables are in lut (-1: none)
  float lut[NLUT];
  float2 sgn2[5];    // (sign_i, sign_i), sign_i = bit_i(lane) ? 1/2 : -1/2

  __device__ __forceinline__ void advance(uint32_t bytes, uint32_t rbytes) {
    o += bytes;
    opos += bytes;
    if (opos >= rbytes) opos -= rbytes;
  }
};

__device__ __forceinline__ void build_lut(const SmemLayout& L, int j, Worker& K) {
  const uint32_t xb = L.xl + j * XL_FLOATS * 4;
#pragma unroll
  for (int p = 0; p < 7; ++p) {
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const float2 xv = lds<float2>(xb + (p * 5 + i) * 8);
      acc = __ffma2_rn(K.sgn2[i], xv, acc);
    }
    K.lut[2 * p] = acc.x;
    if (2 * p + 1 < NLUT) K.lut[2 * p + 1] = acc.y;
  }
  K.lut_col = j;
}

// Loads the 32 X pairs of staging slot j (the same in every lane).
__device__ __forceinline__ void load_xp(const SmemLayout& L, int j, uint32_t (&xp)[32]) {
  const uint32_t base = smem_u32(vbq_smem) + L.X + j * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 v = lds_v4(base + 16 * q);
    xp[4 * q] = v.x;
    xp[4 * q + 1] = v.y;
    xp[4 * q + 2] = v.z;
    xp[4 * q + 3] = v.w;
  }
}

// Decodes U consecutive steps of class CLS with e entries each, the first at
// ring position pos, and adds the entries into the CTA's row accumulators at
// acc_a (the run's super-tile slot). Lane l works on entry l of each step (lanes
// past e of a partial step read entry 0 and add nothing). The first step's
// first entry is entry i0 of the run (its tile comes from the header's prefix
// counts).
template <int CLS, int U>
__device__ __forceinline__ void do_steps(const WarpStream& S, uint32_t pos, uint32_t e, uint32_t i0,
                                         const RunHeader& h, uint32_t acc_a, const Worker& K,
                                         const uint32_t (&xp)[32], const ColInfo& ci, int lane) {
  constexpr uint32_t B = 1u << CLS;
  constexpr uint32_t FULL = full_step_bytes(CLS);
  const uint32_t me = static_cast<uint32_t>(lane) < e ? static_cast<uint32_t>(lane) : 0u;
  const bool lead = static_cast<uint32_t>(lane) < e;
  int iv[U];
  uint32_t row[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint32_t p = pos + u * FULL;
    if (p >= S.rbytes) p -= S.rbytes;
    const uint32_t rec = S.ring + p;
    const uint32_t sb = lds<uint16_t>(rec + rec_scale_off(CLS, e) + 2u * me);
    row[u] = lds<uint8_t>(rec + rec_row_off(CLS, e) + me);
    float v;
    if constexpr (CLS == 0) {
      const uint2 cw = lds<uint2>(rec + 8u * me);
      v = half_bits_to_float(sb) * decode_plane(cw, K.lut);
    } else {
      uint32_t w[16];
#pragma unroll
      for (uint32_t q = 0; q < B / 2; ++q) {
        const uint4 c = lds_v4(smem_u32(vbq_smem) + rec + (q * e + me) * 16u);
        w[4 * q] = c.x;
        w[4 * q + 1] = c.y;
        w[4 * q + 2] = c.z;
        w[4 * q + 3] = c.w;
      }
      const int sum = decode_dp<CLS>(w, xp);
      const int t2 = 2 * sum - static_cast<int>((1u << B) - 1u) * ci.sum_x;
      v = half_bits_to_float(sb) * (static_cast<float>(t2) * ci.u);
    }
    iv[u] = __float2int_rn(v);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (lead) {
      const uint32_t tile = entry_tile(h, i0 + u * 32u + static_cast<uint32_t>(lane));
      red_shared_add_s32(acc_a + (tile * TILE + row[u]) * 4u, iv[u]);
    }
  }
}

// Steps [k, kend) of a run of class CLS (its header h) whose column sits in
// staging slot cj, accumulating into the CTA accumulator at acc_a. Waits for
// and frees ring bytes. Full steps go U at a time.
template <int CLS, int U>
__device__ __forceinline__ void run_steps_cls(const SmemLayout& L, const RunHeader& h, int cj, uint32_t k,
                                              uint32_t kend, uint32_t acc_a, WarpStream& S, Worker& K, int lane) {
  constexpr uint32_t E = STEP_LANES;
  constexpr uint32_t FULL = full_step_bytes(CLS);
  const uint32_t n = h.n;
  const uint32_t nfull = n >> 5;
  const uint32_t e_last = n - nfull * E;
  uint32_t xp[32];
  ColInfo ci{0, 0.0f};
  if constexpr (CLS == 0) {
    if (K.lut_col != cj) build_lut(L, cj, K);
  } else {
    load_xp(L, cj, xp);
    ci = lds<ColInfo>(L.col + cj * 8);
  }
  if constexpr (U > 1) {
    const uint32_t kf = min(kend, nfull);
    while (k + U <= kf) {
      const uint32_t need = K.o + U * FULL;
      if (S.avail < need) {
        S.wait_for(need);
        if (!S.ok) return;
      }
      do_steps<CLS, U>(S, K.opos, E, k * E, h, acc_a, K, xp, ci, lane);
      K.advance(U * FULL, S.rbytes);
      k += U;
      S.refill(K.o, lane);
    }
  }
  for (; k < kend; ++k) {
    const uint32_t e = k < nfull ? E : e_last;
    const uint32_t rb = k < nfull ? FULL : rec_bytes(CLS, e);
    if (S.avail < K.o + rb) {
      S.wait_for(K.o + rb);
      if (!S.ok) return;
    }
    do_steps<CLS, 1>(S, K.opos, e, k * E, h, acc_a, K, xp, ci, lane);
    K.advance(rb, S.rbytes);
    S.refill(K.o, lane);
  }
}

__device__ __forceinline__ void run_steps_any(const SmemLayout& L, const RunHeader& h, int cj, uint32_t k,
                                              uint32_t kend, uint32_t acc_a, WarpStream& S, Worker& K, int lane) {
  switch (h.cls) {
    case 0: run_steps_cls<0, kU1>(L, h, cj, k, kend, acc_a, S, K, lane); break;
    case 1: run_steps_cls<1, kUdp>(L, h, cj, k, kend, acc_a, S, K, lane); break;
    case 2: run_steps_cls<2, kUdp>(L, h, cj, k, kend, acc_a, S, K, lane); break;
    default: run_steps_cls<3, kUdp>(L, h, cj, k, kend, acc_a, S, K, lane); break;
  }
}

// One warp's part of one item: its sub-ranges of the plan (in global or
// shared memory), accumulated into the CTA's accumulators (slot = item
// super-tile - cp.st_base). seg_st_off[s] is the first item super-tile of
// segment s (null: one segment at 0).
__device__ __forceinline__ void warp_item(const SmemLayout& L, const WarpPlan* wp_g, const uint32_t* seg_st_off,
                                          const CtaPlan& cp, WarpStream& S, Worker& K, int lane) {
  const uint32_t nsub = wp_g->nsub;
  for (uint32_t si = 0; si < nsub && S.ok; ++si) {
    const SubRange* sp = &wp_g->sub[si];
    RunHeader h;
    {
      const uint4 hv = *reinterpret_cast<const uint4*>(&sp->first);
      h = *reinterpret_cast<const RunHeader*>(&hv);
    }
    uint32_t k = sp->k0;
    uint32_t left = sp->nsteps;
    const uint32_t soff = seg_st_off ? seg_st_off[sp->seg] : 0u;
    if (left == 0) continue;
    if (k == 0) K.advance(HEADER_BYTES, S.rbytes);  // the range starts at the run's header, which the warp has
    while (true) {
      const uint32_t nrs = run_steps(h.cls, h.n);
      const uint32_t kend = min(nrs, k + left);
      const uint32_t slot = soff + h.row0 / SROWS - cp.st_base;
      const uint32_t acc_a = smem_u32(vbq_smem) + L.acc + slot * (SROWS * 4u);
      run_steps_any(L, h, static_cast<int>(col_slot(cp, h.g)), k, kend, acc_a, S, K, lane);
      if (!S.ok) return;
      left -= kend - k;
      if (left == 0) break;
      // The next run of the range: its header comes from the stream.
      if (S.avail < K.o + HEADER_BYTES) {
        S.wait_for(K.o + HEADER_BYTES);
        if (!S.ok) return;
      }
      const uint4 hv = lds_v4(S.ring_a + K.opos);
      h = *reinterpret_cast<const RunHeader*>(&hv);
      K.advance(HEADER_BYTES, S.rbytes);
      S.refill(K.o, lane);
      k = 0;
    }
  }
}

__device__ __forceinline__ void worker_init(WarpStream& S, Worker& K, const SmemLayout& L, uint32_t ns,
                                            const uint64_t* pieces, const uint32_t* pstart, const uint32_t* pbytes,
                                            int lane, int warp) {
  const size_t wi = static_cast<size_t>(blockIdx.x) * KW + warp;
  const uint32_t p0 = pstart[wi], p1 = pstart[wi + 1];
  S.init(L.ring + warp * L.ring_stride, ns, smem_u32(vbq_smem) + L.bar + warp * NS_MAX * 8, pieces + p0, p1 - p0,
         pbytes[wi], lane);
  S.start(lane);
  K.o = 0;
  K.opos = 0;
  K.lut_col = -1;
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const float sg = ((lane >> i) & 1) ? 0.5f : -0.5f;
    K.sgn2[i] = make_float2(sg, sg);
  }
#pragma unroll
  for (int k = 0; k < NLUT; ++k) K.lut[k] = 0.0f;
}

// Adds the CTA's row accumulators of its slots into the fixed-point output
// out [item rows] and clears them. All threads.
__device__ __forceinline__ void flush_slots(const SmemLayout& L, const CtaPlan& cp, unsigned long long* out) {
  const uint32_t total = cp.n_slots * SROWS;
  for (uint32_t i = threadIdx.x; i < total; i += KW * 32) {
    const int v = lds<int>(L.acc + 4 * i);
    if (v != 0) {
      red_add_u64(out + static_cast<size_t>(cp.st_base) * SROWS + i, static_cast<long long>(v));
      sts<int>(L.acc + 4 * i, 0);
    }
  }
}

// Max |x| over K bf16 values (all threads of the CTA; every CTA gets the same value).
__device__ __forceinline__ float max_abs_bf16(const uint16_t* x, int K, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = 0.0f;
  constexpr int PER = (XCAP / 2 + KW * 32 - 1) / (KW * 32);  // u32 pairs per thread at most
  uint32_t v[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int i = threadIdx.x + j * KW * 32;
    v[j] = 2 * i < K ? ldg_nc_u32(x + 2 * i) : 0u;
  }
#pragma unroll
  for (int j = 0; j < PER; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(v[j])), fabsf(bf16_hi(v[j]))));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < KW; ++w) r = fmaxf(r, red[w]);
  return r;
}

}  // namespace vbq
