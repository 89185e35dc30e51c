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

constexpr int CH = 4096;             // bytes per bulk copy and per ring slot
constexpr int LOG_CH = 12;
constexpr int NS_MAX = 6;            // ring slots per warp at most
constexpr int SPILL = 512;           // bytes past the ring's end (>= header + the largest record)
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
#define VBQ_UDP 2
#endif
constexpr int kRingSlots = VBQ_NS;
constexpr int kU1 = VBQ_U1;
constexpr int kUdp = VBQ_UDP;
static_assert(kRingSlots >= 2 && kRingSlots <= 6, "ring slots");

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

// Stores a column into staging slot j: lane l gives x_{2l} and x_{2l+1} (bf16
// values held in floats). Whole warp. F is the fixed-point exponent.
__device__ __forceinline__ void put_column(const SmemLayout& L, int j, float x0, float x1, int F, int lane) {
  float m = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  int s = 0;
  if (m > 0.0f) {
    int e;
    frexpf(m, &e);  // m < 2^e, so |x| * 2^(14 - e) < 2^14
    s = 14 - e;
  }
  const int X0 = __float2int_rn(scalbnf(x0, s)), X1 = __float2int_rn(scalbnf(x1, s));
  int sx = X0 + X1;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, d);
  sts<uint32_t>(L.X + j * 128 + 4 * lane, (static_cast<uint32_t>(X0) & 0xFFFFu) | (static_cast<uint32_t>(X1) << 16));
  // Lookup order: float2 (x'_{10p+i}, x'_{10p+5+i}) at pair p*5 + i, p = 0..6, i = 0..4, x' = x * 2^F.
  const uint32_t xb = L.xl + j * XL_FLOATS * 4;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int jj = 2 * lane + h;
    const int p = jj / 10, w = jj - 10 * p;
    const int idx = (p * 5 + (w % 5)) * 2 + w / 5;
    sts<float>(xb + idx * 4, scalbnf(h ? x1 : x0, F));
  }
  // x_64 .. x_69 do not exist: zero their slots (indices 68 and 61, 63, 65, 67, 69).
  if (lane < 6) sts<float>(xb + (lane == 0 ? 68 : 59 + 2 * lane) * 4, 0.0f);
  if (lane == 0) {
    ColInfo ci;
    ci.sum_x = sx;
    ci.u = scalbnf(1.0f, F - s - 1);
    sts<ColInfo>(L.col + j * 8, ci);
  }
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

// sum q X over the lane's slice of a 2-, 4- or 8-bit entry (exact int32).
template <int CLS>
__device__ __forceinline__ int decode_dp(uint2 cw, const uint32_t (&xp)[16]) {
  int s = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t w = h ? cw.y : cw.x;
    if constexpr (CLS == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t by = (w >> (2 * i)) & 0x03030303u;
        s = dp2a_lo(xp[8 * h + 2 * i], by, s);
        s = dp2a_hi(xp[8 * h + 2 * i + 1], by, s);
      }
    } else if constexpr (CLS == 2) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t by = (w >> (4 * i)) & 0x0F0F0F0Fu;
        s = dp2a_lo(xp[4 * h + 2 * i], by, s);
        s = dp2a_hi(xp[4 * h + 2 * i + 1], by, s);
      }
    } else {
      s = dp2a_lo(xp[2 * h], w, s);
      s = dp2a_hi(xp[2 * h + 1], w, s);
    }
  }
  return s;
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

// Loads the lane's X pairs of staging slot j for class CLS (lane slice s = lane & (b - 1)).
template <int CLS>
__device__ __forceinline__ void load_xp(const SmemLayout& L, int j, int lane, uint32_t (&xp)[16]) {
  constexpr int B = 1 << CLS;
  constexpr int NP = 32 / B;  // int16 pairs in the slice
  const uint32_t base = L.X + j * 128 + (lane & (B - 1)) * (128 / B);
#pragma unroll
  for (int q = 0; q < NP / 4; ++q) {
    const uint4 v = lds_v4(smem_u32(vbq_smem) + base + 16 * q);
    xp[4 * q] = v.x;
    xp[4 * q + 1] = v.y;
    xp[4 * q + 2] = v.z;
    xp[4 * q + 3] = v.w;
  }
}

// Decodes U consecutive steps of class CLS with e entries each, the first at
// ring position pos, and adds the entries into the CTA's row accumulators at
// acc_a (the run's super-tile slot). The first step's first entry is entry i0
// of the run (its tile comes from the header's prefix counts).
template <int CLS, int U>
__device__ __forceinline__ void do_steps(const WarpStream& S, uint32_t pos, uint32_t e, uint32_t i0,
                                         const RunHeader& h, uint32_t acc_a, const Worker& K,
                                         const uint32_t (&xp)[16], const ColInfo& ci, int lane) {
  constexpr uint32_t B = 1u << CLS;
  constexpr uint32_t E = 32u >> CLS;
  constexpr uint32_t FULL = full_step_bytes(CLS);
  const uint32_t j = static_cast<uint32_t>(lane) >> CLS;
  const uint32_t sigma = static_cast<uint32_t>(lane) & (B - 1u);
  const uint32_t me = CLS == 0 ? static_cast<uint32_t>(lane) : j;  // the entry whose scale and row this lane reads
  const bool lead = (CLS == 0 ? static_cast<uint32_t>(lane) < e : (sigma == 0 && j < e));
  uint2 cw[U];
  uint32_t sb[U], row[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    uint32_t p = pos + u * FULL;
    if (p >= S.rbytes) p -= S.rbytes;
    const uint32_t rec = S.ring + p;
    cw[u] = lds<uint2>(rec + 8u * lane);
    sb[u] = lds<uint16_t>(rec + rec_scale_off(CLS, e) + 2u * me);
    row[u] = lds<uint8_t>(rec + rec_row_off(CLS, e) + me);
  }
  int iv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float v;
    if constexpr (CLS == 0) {
      v = half_bits_to_float(sb[u]) * decode_plane(cw[u], K.lut);
    } else {
      int s = decode_dp<CLS>(cw[u], xp);
#pragma unroll
      for (uint32_t d = 1; d < B; d <<= 1) s += __shfl_xor_sync(0xffffffffu, s, static_cast<int>(d));
      const int t2 = 2 * s - static_cast<int>((1u << B) - 1u) * ci.sum_x;
      v = half_bits_to_float(sb[u]) * (static_cast<float>(t2) * ci.u);
    }
    iv[u] = __float2int_rn(v);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (lead) {
      const uint32_t tile = entry_tile(h, i0 + u * E + me);
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
  constexpr uint32_t E = 32u >> CLS;
  constexpr uint32_t FULL = full_step_bytes(CLS);
  const uint32_t n = h.n;
  const uint32_t nfull = n >> (5 - CLS);
  const uint32_t e_last = n - nfull * E;
  uint32_t xp[16];
  ColInfo ci{0, 0.0f};
  if constexpr (CLS == 0) {
    if (K.lut_col != cj) build_lut(L, cj, K);
  } else {
    load_xp<CLS>(L, cj, lane, xp);
    ci = lds<ColInfo>(L.col + cj * 8);
  }
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

// One warp's part of one item: its sub-ranges of the plan, accumulated into
// the CTA's accumulators (slot = item super-tile - cp.st_base). seg_st_off[s]
// is the first item super-tile of segment s (null: one segment at 0).
__device__ __forceinline__ void warp_item(const SmemLayout& L, const WarpPlan* wp_g, const uint32_t* seg_st_off,
                                          const CtaPlan& cp, WarpStream& S, Worker& K, int lane) {
  const uint32_t nsub = __ldg(&wp_g->nsub);
  for (uint32_t si = 0; si < nsub && S.ok; ++si) {
    const SubRange* sp = &wp_g->sub[si];
    RunHeader h;
    {
      const uint4 hv = __ldg(reinterpret_cast<const uint4*>(&sp->first));
      h = *reinterpret_cast<const RunHeader*>(&hv);
    }
    uint32_t k = __ldg(&sp->k0);
    uint32_t left = __ldg(&sp->nsteps);
    const uint32_t soff = seg_st_off ? seg_st_off[__ldg(&sp->seg)] : 0u;
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
