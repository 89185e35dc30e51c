// Dequant-MMA for batches of 2..64 columns: Y = W X on the 5th-generation
// tensor cores (tcgen05), one launch for all columns.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): the packed per-group
// codes are dequantized and multiplied in one pass. With two or more
// activation columns the product is a dense contraction, so this kernel
// rebuilds W as fp16 in shared memory, one (256-row tile, group column) at a
// time, and feeds it to tcgen05.mma. The design is this library's own:
//
//  * Work: the (tile, group column) pairs in tile-major order are cut into
//    contiguous ranges of about equal cost, one range per CTA (one CTA per
//    SM). A tile whose columns span several CTAs adds their partial sums in
//    CTA order (fixed, so results do not depend on timing); the last of its
//    CTAs to finish does the sum, with many loads in flight per thread.
//  * Stream: a pair's data are, for each bit class, the steps of the class's
//    run (layout.h) that hold the tile's entries: at most four pieces, copied
//    with cp.async.bulk into one of four shared-memory stages. Every wait is
//    bounded. The column scales, the B tiles and this kernel are three
//    launches chained as programmatic dependents, so each starts while the one
//    before finishes.
//  * Dequant: a warp takes one 32-code block of a 32-entry step at a time,
//    lane l entry l, and writes that part of the entry's row of
//    A = s_g * (q - c_b), rounded once to fp16, into a 256 x 64 K-major tile
//    with the 128-byte swizzle (two 128-row halves). Inside each 32-code
//    block of a group, K position 2s + h holds code s + 16h (s < 16): a 1-bit
//    word yields the pair as the pattern of -s/2 with one shift and one
//    sign flip, a 2-, 4- or 8-bit entry with a mask per word and one byte
//    permute. The blocks of a pair are dealt to the warps in turn, continuing
//    from pair to pair, so that no warp always gets a pair's leftovers.
//    B is the same group of each batch column, times a per-column power of two
//    that keeps it inside fp16's range, in the same order; the product does
//    not depend on the order of K.
//  * MMA: one thread issues tcgen05.mma.cta_group::1.kind::f16 (M = 128,
//    N = batch rounded up to 16, K = 16; four K-steps per half) into fp32
//    accumulators in tensor memory and commits to an mbarrier. A and B are
//    double-buffered, so the warps dequantize the next pair while the tensor
//    cores run.
//  * Epilogue: tcgen05.ld of each warp's 32-lane quadrant, divided by the
//    column's power of two.
// Exactness: each weight is rounded once to fp16 (relative error <= 2^-11),
// x once to fp16 after an exact power-of-two scaling, and the products are
// summed in fp32. Scales above 512 would overflow fp16 (|q - c| <= 127.5);
// such matrices take the CUDA-core path.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace vbq {

extern __shared__ __align__(1024) uint8_t tc_smem[];

namespace {

#ifndef VBQ_TC_DEQ
#define VBQ_TC_DEQ 16
#endif
constexpr int TC_DEQ = VBQ_TC_DEQ;       // dequant warps (a multiple of 8: the epilogue's quadrants)
static_assert(TC_DEQ % 8 == 0 && TC_DEQ >= 8, "dequant warps");
constexpr int TC_WARPS = TC_DEQ + 2;     // and a copy warp and an MMA warp
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int TC_NMAX = 64;              // batch columns per launch
constexpr int TC_BTILE = TC_NMAX * 128;  // fp16 B tile: 64 columns x 64 K
constexpr int TC_PIECE_BYTES = 24576;    // bytes of one pair's pieces at most
constexpr int TC_STAGE = TC_BTILE + TC_PIECE_BYTES;  // a stage: the pair's B tile, then its pieces
constexpr int TC_NST = 4;                // stages
constexpr int TC_MAX_PIECES = 1024;      // pieces of one CTA
constexpr int TC_MAX_PAIRS = 512;        // pairs of one CTA
constexpr int TC_MAX_UNITS = 64;         // tiles of one CTA
constexpr int TC_ATILE = 256 * 128;      // fp16 A tile: 256 rows x 64 K
constexpr float TC_MAX_SCALE = 512.0f;

// The steps of one class run that hold one tile's entries of one group column.
struct TcPiece {      // 16 bytes
  uint32_t off16;     // first byte of the first step, / 16, from the matrix data
  uint16_t bytes16;   // bytes / 16
  uint8_t cls;
  uint8_t nst;        // steps
  uint16_t n;         // entries of the run
  uint16_t ks;        // run step of the first step
  uint16_t lo, hi;    // the tile's entries [lo, hi) of the run
};
static_assert(sizeof(TcPiece) == 16, "piece record");

// One tile's group columns inside one CTA.
struct TcUnit {
  uint32_t tile;
  uint32_t p0, p1;    // pairs [p0, p1), pair = tile * G + g
  uint32_t pbase;     // first partial block of the tile (split tiles)
  uint16_t split, nsplit;
};

struct TcCta {
  uint32_t u0, u1;    // units
  uint32_t q0, q1;    // pieces
};

struct TcSmem {
  static constexpr int kA = 0;                                  // [2][256 x 128 B], 1024-aligned
  static constexpr int kStage = kA + 2 * TC_ATILE;              // [TC_NST][TC_STAGE], 1024-aligned
  static constexpr int kPiece = kStage + TC_NST * TC_STAGE;     // TcPiece [TC_MAX_PIECES]
  static constexpr int kPair = kPiece + TC_MAX_PIECES * 16;     // first piece of each pair, [TC_MAX_PAIRS + 1]
  static constexpr int kUnit = kPair + (TC_MAX_PAIRS + 1) * 4 + 12;  // TcUnit [TC_MAX_UNITS]
  static constexpr int kSx = kUnit + TC_MAX_UNITS * sizeof(TcUnit);  // per batch column scale
  static constexpr int kBar = kSx + TC_NMAX * 4;                // mbarriers: 2 per stage, 8 more
  static constexpr int kMisc = kBar + 8 * (2 * TC_NST + 10);
  static constexpr int kBytes = kMisc + 64 + 1024;  // + room to align the tiles to 1024 bytes
};
static_assert(TcSmem::kBar % 8 == 0 && TC_STAGE % 1024 == 0, "alignment of the mbarriers and the B tiles");
static_assert(TcSmem::kBytes <= 232448, "shared memory of the tensor-core kernel");

struct TcArgs {
  const uint8_t* data;
  const TcCta* ctas;
  const TcUnit* units;
  const TcPiece* pieces;
  const uint32_t* pair_piece;   // [n_pairs + 1]
  float* partial;               // [split blocks][TC_NMAX][256]
  uint32_t* counters;           // per split tile
  const uint8_t* bt;            // [G][TC_NMAX x 128 B]: each group's B tile, as laid out in shared memory
  const float* sx;              // [B] powers of two
  float* Y;                     // [B][N]
  int32_t B, Npad, K, G;
  int64_t N;
  int* err;
};

// Element chunk (row, chunk) of an 8-row-atom, 128-byte-swizzled, K-major tile.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// fp16 pairs without conversions: 0x6400 | q is the fp16 value 1024 + q
// (q < 1024). With c = (2^b - 1)/2 = m0 + 1/2, (1024 + q) - (1024 + m0) = q - m0
// exactly, and fma(q - m0, s, -s/2) = s * (q - c) rounded once (s/2 is exact in
// fp16 for the scales this path takes).
__device__ __forceinline__ uint32_t deq_pair(uint32_t h1024q, __half2 base, __half2 sc, __half2 nhs) {
  const __half2 v = __hfma2(__hsub2(*reinterpret_cast<const __half2*>(&h1024q), base), sc, nhs);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void put16(uint32_t a_base, uint32_t row, uint32_t chunk, uint4 v) {
  *reinterpret_cast<uint4*>(tc_smem + a_base + (row >> 7) * (TC_ATILE / 2) + sw128(row & 127u, chunk)) = v;
}

// Dequantizes block blk (codes 32 blk .. 32 blk + 31) of entry `lane` of a
// step of class CLS (e entries) at shared offset rec into its row of A, if the
// entry is one of the tile's. Inside the block, K position 2s + h holds code
// s + 16h (s < 16), four pairs per 16-byte chunk.
template <int CLS>
__device__ __forceinline__ void tc_entry(uint32_t rec, uint32_t e, bool mine, uint32_t blk, uint32_t a_base, int lane) {
  constexpr uint32_t B = 1u << CLS;
  if (!mine) return;
  const uint32_t j = static_cast<uint32_t>(lane);
  const uint16_t sb = *reinterpret_cast<const uint16_t*>(tc_smem + rec + rec_scale_off(CLS, e) + 2u * j);
  const uint32_t row = tc_smem[rec + rec_row_off(CLS, e) + j];
  if constexpr (CLS == 0) {
    // w = s (q - 1/2) = -+s/2: the fp16 pattern of -s/2, its sign flipped where
    // q = 1 (the same two values the fma form gives when s/2 is exact).
    const uint32_t w = *reinterpret_cast<const uint32_t*>(tc_smem + rec + 8u * j + 4u * blk);
    const __half hs = __hmul(__ushort_as_half(sb), __float2half_rn(0.5f));
    const uint32_t neg = static_cast<uint32_t>(__half_as_ushort(hs)) ^ 0x8000u;
    const uint32_t pat = neg | (neg << 16);
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c) {  // chunk 4 blk + c: pairs s = 4c .. 4c + 3
      uint32_t o[4];
#pragma unroll
      for (uint32_t t = 0; t < 4; ++t) {
        const uint32_t sh = 4u * c + t;                       // code sh at bit 15, code sh + 16 at bit 31
        o[t] = pat ^ ((w << (15u - sh)) & 0x80008000u);
      }
      put16(a_base, row, 4u * blk + c, make_uint4(o[0], o[1], o[2], o[3]));
    }
  } else {
    const __half2 sc = __half2half2(__ushort_as_half(sb));
    const __half2 nhs = __hmul2(sc, __float2half2_rn(-0.5f));
    const __half2 base = __float2half2_rn(static_cast<float>(1024u + (1u << (B - 1u)) - 1u));
    // The block's B words (blk*B .. blk*B + B - 1), 16-byte chunk q of entry j at 16 (q e + j).
    uint32_t w[B];
    if constexpr (B == 2) {
      const uint4 v = *reinterpret_cast<const uint4*>(tc_smem + rec + j * 16u);
      w[0] = blk ? v.z : v.x;
      w[1] = blk ? v.w : v.y;
    } else {
#pragma unroll
      for (uint32_t q = 0; q < B / 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(tc_smem + rec + ((blk * B / 4 + q) * e + j) * 16u);
        w[4 * q] = v.x;
        w[4 * q + 1] = v.y;
        w[4 * q + 2] = v.z;
        w[4 * q + 3] = v.w;
      }
    }
    constexpr uint32_t CPW = 32u / B;              // codes per word
    constexpr uint32_t MASK = B == 8 ? 0xFFFFFFFFu : (B == 4 ? 0x0F0F0F0Fu : 0x03030303u);
    // Code s (< 16) of the block is code s % CPW of word s / CPW, and code s + 16
    // the same code of the word B/2 further on.
#pragma unroll
    for (uint32_t u = 0; u < B / 2; ++u) {
      const uint32_t wa = w[u], wb = w[u + B / 2];
#pragma unroll
      for (uint32_t i = 0; i < CPW / 4; ++i) {
        const uint32_t va = (wa >> (B * i)) & MASK, vb = (wb >> (B * i)) & MASK;
        uint32_t o[4];
#pragma unroll
        for (uint32_t t = 0; t < 4; ++t) {
          const uint32_t pr = __byte_perm(va, vb, t | (t << 4) | ((4u + t) << 8) | ((4u + t) << 12));
          o[t] = deq_pair((pr & 0x00FF00FFu) | 0x64006400u, base, sc, nhs);
        }
        // pairs s = u * CPW + 4i .. + 3: chunk (u * CPW + 4i) / 4 of the block
        put16(a_base, row, 4u * blk + u * (CPW / 4) + i, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
}

__device__ __forceinline__ void tc_step(uint32_t rec, uint32_t cls, uint32_t e, bool mine, uint32_t blk,
                                        uint32_t a_base, int lane) {
  switch (cls) {
    case 0: tc_entry<0>(rec, e, mine, blk, a_base, lane); break;
    case 1: tc_entry<1>(rec, e, mine, blk, a_base, lane); break;
    case 2: tc_entry<2>(rec, e, mine, blk, a_base, lane); break;
    default: tc_entry<3>(rec, e, mine, blk, a_base, lane); break;
  }
}

// Roles: warps 0 .. TC_DEQ-1 dequantize (and run the epilogue), warp TC_DEQ
// copies (one lane), warp TC_DEQ+1 issues the MMAs (one lane). They hand work
// over through mbarriers only:
//   stage_full[s]  the pair's B tile and pieces have landed (copy bytes)
//   stage_empty[s] the pair's MMAs are done, so its stage may be refilled (commit)
//   a_full[b]      every dequant warp has written its rows of A buffer b (TC_DEQ arrivals)
//   a_empty[b]     the MMAs that read A buffer b are done (commit)
//   acc_full[t]    the unit's MMAs into accumulator t are done (commit)
//   acc_empty[t]   the epilogue has read accumulator t (TC_DEQ arrivals)
// A wait that runs out sets the shared abort flag; every role then stops at
// its next wait, and the CTA waits (bounded) for its copies and MMAs in flight.
__global__ void __launch_bounds__(TC_THREADS, 1) vbq_gemm_tc_kernel(const __grid_constant__ TcArgs a) {
  using L = TcSmem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Every region sits at its offset from the first 1024-byte boundary of the dynamic shared memory.
  const uint32_t sraw = smem_u32(tc_smem);
  const uint32_t pad = ((sraw + 1023u) & ~1023u) - sraw;
  const uint32_t sbase = sraw + pad;
  uint8_t* const sm = tc_smem + pad;
  TcPiece* pcs = reinterpret_cast<TcPiece*>(sm + L::kPiece);
  uint32_t* pfirst = reinterpret_cast<uint32_t*>(sm + L::kPair);
  TcUnit* units = reinterpret_cast<TcUnit*>(sm + L::kUnit);
  float* sxs = reinterpret_cast<float*>(sm + L::kSx);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + L::kMisc);  // [0] TMEM, [1] abort, [2] last
  const uint32_t bar_sf = sbase + L::kBar;               // stage_full [TC_NST]
  const uint32_t bar_se = bar_sf + 8 * TC_NST;           // stage_empty [TC_NST]
  const uint32_t bar_af = bar_se + 8 * TC_NST;           // a_full [2]
  const uint32_t bar_ae = bar_af + 16;                   // a_empty [2]
  const uint32_t bar_cf = bar_ae + 16;                   // acc_full [2]
  const uint32_t bar_ce = bar_cf + 16;                   // acc_empty [2]
  const uint32_t bar_ed = bar_ce + 16;                   // epi_done (split tiles)
  const uint32_t bar_dc = bar_ed + 8;                    // decided (split tiles)
  const uint32_t N = static_cast<uint32_t>(a.Npad);

  const TcCta cta = a.ctas[blockIdx.x];
  const uint32_t nu = cta.u1 - cta.u0;
  if (nu == 0) return;
  for (uint32_t i = tid; i < nu; i += TC_THREADS) units[i] = a.units[cta.u0 + i];
  for (uint32_t i = tid; i < cta.q1 - cta.q0; i += TC_THREADS) pcs[i] = a.pieces[cta.q0 + i];
  const uint32_t pa = a.units[cta.u0].p0, pb = a.units[cta.u1 - 1].p1;  // the CTA's pairs
  for (uint32_t i = tid; i <= pb - pa; i += TC_THREADS) pfirst[i] = a.pair_piece[pa + i] - cta.q0;
  grid_dep_wait();  // the B tiles and column scales of the kernels before are complete
  for (int i = tid; i < TC_NMAX; i += TC_THREADS) sxs[i] = i < a.B ? a.sx[i] : 0.0f;
  if (tid == 0) {
    for (int i = 0; i < TC_NST; ++i) {
      mbar_init(bar_sf + 8 * i, 1);
      mbar_init(bar_se + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_af + 8 * i, TC_DEQ);
      mbar_init(bar_ae + 8 * i, 1);
      mbar_init(bar_cf + 8 * i, 1);
      mbar_init(bar_ce + 8 * i, TC_DEQ);
    }
    mbar_init(bar_ed, TC_DEQ);
    mbar_init(bar_dc, 1);
    misc[1] = 0u;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + L::kMisc, 4 * TC_NMAX);  // 256 columns: two accumulators of two 128-lane halves of N <= 64
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t npairs = pb - pa;
  auto abort_now = [&]() { misc[1] = 1u; };
  auto aborted = [&]() { return misc[1] != 0u; };

  if (warp == TC_DEQ) {
    // ---- producer: pair i's B tile and pieces into stage i % TC_NST ----
    if (lane == 0) {
      uint32_t i = 0;
      for (; i < npairs; ++i) {
        const uint32_t s = i % TC_NST;
        if (i >= static_cast<uint32_t>(TC_NST)) {
          if (aborted() || !mbar_wait(bar_se + 8 * s, ((i / TC_NST) - 1u) & 1u)) {
            abort_now();
            break;
          }
        }
        const uint32_t stg = sbase + L::kStage + s * TC_STAGE;
        fence_proxy_async_smem();
        uint32_t bytes = N * 128u;
        for (uint32_t q = pfirst[i]; q < pfirst[i + 1]; ++q) bytes += 16u * pcs[q].bytes16;
        mbar_arrive_expect_tx(bar_sf + 8 * s, bytes);
        const uint32_t g = (pa + i) % static_cast<uint32_t>(a.G);
        bulk_g2s_plain(stg, a.bt + static_cast<size_t>(g) * TC_BTILE, N * 128u, bar_sf + 8 * s);
        uint32_t o = TC_BTILE;
        for (uint32_t q = pfirst[i]; q < pfirst[i + 1]; ++q) {
          const uint32_t nb = 16u * pcs[q].bytes16;
          bulk_g2s_plain(stg + o, a.data + static_cast<uint64_t>(pcs[q].off16) * 16u, nb, bar_sf + 8 * s);
          o += nb;
        }
      }
      // Copies still in flight land before the CTA may exit: wait (bounded) for the last fills.
      for (uint32_t j = (i > static_cast<uint32_t>(TC_NST) ? i - TC_NST : 0u); j < i; ++j)
        (void)mbar_wait(bar_sf + 8 * (j % TC_NST), (j / TC_NST) & 1u);
    }
  } else if (warp == TC_DEQ + 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      const uint32_t idesc = tc_idesc_f16(128, N);
      uint32_t gi = 0;
      bool ok = true;
      for (uint32_t u = 0; u < nu && ok; ++u) {
        const TcUnit un = units[u];
        const uint32_t rows = static_cast<uint32_t>(a.N - static_cast<int64_t>(un.tile) * 256 < 256
                                                        ? a.N - static_cast<int64_t>(un.tile) * 256 : 256);
        const uint32_t acc = tmem + (u & 1u) * (2u * TC_NMAX);
        if (u >= 2 && (aborted() || !mbar_wait(bar_ce + 8 * (u & 1u), ((u >> 1) - 1u) & 1u))) {
          ok = false;
          break;
        }
        for (uint32_t p = un.p0; p < un.p1; ++p, ++gi) {
          const uint32_t s = gi % TC_NST, buf = gi & 1u;
          if (aborted() || !mbar_wait(bar_af + 8 * buf, (gi >> 1) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = sbase + L::kA + buf * TC_ATILE;
          const uint32_t b_addr = sbase + L::kStage + s * TC_STAGE;
          for (uint32_t h = 0; h < (rows > 128u ? 2u : 1u); ++h) {
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint64_t ad = tc_desc_sw128(a_addr + h * (TC_ATILE / 2) + kk * 32u, 1024u);
              const uint64_t bd = tc_desc_sw128(b_addr + kk * 32u, 1024u);
              tc_mma_f16(acc + h * N, ad, bd, idesc, p > un.p0 || kk > 0);
            }
          }
          tc_commit(bar_ae + 8 * buf);
          tc_commit(bar_se + 8 * s);
          if (p + 1 == un.p1) tc_commit(bar_cf + 8 * (u & 1u));
        }
      }
      if (!ok) abort_now();
      // The MMAs in flight finish before the CTA may exit.
      if (gi > 0) (void)mbar_wait(bar_ae + 8 * ((gi - 1u) & 1u), ((gi - 1u) >> 1) & 1u);
    }
  } else {
    // ---- dequant warps, then the epilogue of each unit ----
    uint32_t gi = 0, su = 0, ibase = 0;  // pairs, split units and work items of this CTA so far
    bool ok = true;
    for (uint32_t u = 0; u < nu && ok; ++u) {
      const TcUnit un = units[u];
      const int64_t r0 = static_cast<int64_t>(un.tile) * 256;
      const uint32_t rows = static_cast<uint32_t>(a.N - r0 < 256 ? a.N - r0 : 256);
      for (uint32_t p = un.p0; p < un.p1; ++p, ++gi) {
        const uint32_t s = gi % TC_NST, buf = gi & 1u;
        bool w = !aborted();
        if (w && gi >= 2) w = mbar_wait(bar_ae + 8 * buf, ((gi >> 1) - 1u) & 1u);
        if (w) w = mbar_wait(bar_sf + 8 * s, (gi / TC_NST) & 1u);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        const uint32_t a_base = L::kA + buf * TC_ATILE + pad;
        // Work items: two per step (its two 32-code blocks), numbered in piece order
        // across the CTA's pairs; warp w takes the items numbered w mod TC_DEQ, so
        // a pair's leftover items fall to different warps from pair to pair.
        uint32_t o = L::kStage + s * TC_STAGE + pad + TC_BTILE;
        for (uint32_t q = pfirst[gi]; q < pfirst[gi + 1]; ++q) {
          const TcPiece pc = pcs[q];
          const uint32_t fb = full_step_bytes(pc.cls);
          const uint32_t nit = 2u * pc.nst;
          uint32_t it = (static_cast<uint32_t>(warp) + TC_DEQ - ibase % TC_DEQ) % TC_DEQ;
          for (; it < nit; it += TC_DEQ) {
            const uint32_t k = it >> 1, blk = it & 1u;
            const uint32_t k0 = 32u * (pc.ks + k);
            const uint32_t e = min(32u, static_cast<uint32_t>(pc.n) - k0);
            const uint32_t i = k0 + static_cast<uint32_t>(lane);
            const bool mine = static_cast<uint32_t>(lane) < e && i >= pc.lo && i < pc.hi;
            tc_step(o + k * fb, pc.cls, e, mine, blk, a_base, lane);
          }
          ibase += nit;
          o += 16u * pc.bytes16;
        }
        fence_proxy_async_smem();  // this warp's rows of A, for the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_af + 8 * buf);
      }
      if (!ok) break;

      // ---- epilogue of unit u ----
      if (aborted() || !__all_sync(0xffffffffu, mbar_wait(bar_cf + 8 * (u & 1u), (u >> 1) & 1u))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Warp w reads TMEM lanes 32 (w % 4) .. + 31 of half (w / 4) % 2, column blocks 16 (w / 8), + 32, ...
      const uint32_t acc = tmem + (u & 1u) * (2u * TC_NMAX);
      const uint32_t quad = static_cast<uint32_t>(warp & 3), half = static_cast<uint32_t>((warp >> 2) & 1);
      const uint32_t r = half * 128u + quad * 32u + static_cast<uint32_t>(lane);
      float* part = un.nsplit > 1 ? a.partial + (static_cast<size_t>(un.pbase) + un.split) * (TC_NMAX * 256) : nullptr;
      if (half == 0 || rows > 128u) {
        for (uint32_t c0 = 16u * static_cast<uint32_t>(warp >> 3); c0 < N; c0 += 16u * (TC_DEQ / 8)) {
          uint32_t v[16];
          tmem_ld16(acc + ((quad * 32u) << 16) + half * N + c0, v);
          tmem_ld_wait();
          if (r < rows) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t bc = c0 + static_cast<uint32_t>(i);
              if (bc < static_cast<uint32_t>(a.B)) {
                const float y = __uint_as_float(v[i]) / sxs[bc];
                if (part) part[bc * 256u + r] = y;
                else a.Y[static_cast<int64_t>(bc) * a.N + r0 + r] = y;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ce + 8 * (u & 1u));  // the accumulator may be overwritten
      if (un.nsplit > 1) {
        // The last of the tile's CTAs adds the partial blocks in split order. The
        // dequant warps meet on mbarriers (bounded waits): epi_done gathers their
        // partial rows for thread 0's arrival on the tile's counter (a release at
        // GPU scope), and decided hands its answer back.
        if (lane == 0) mbar_arrive(bar_ed);
        bool w = true;
        if (tid == 0) {
          w = mbar_wait(bar_ed, su & 1u);
          misc[2] = w && (atom_add_acq_rel_u32(a.counters + un.tile, 1u) + 1u == un.nsplit) ? 1u : 0u;
          mbar_arrive(bar_dc);
        }
        w = w && mbar_wait(bar_dc, su & 1u);
        ++su;
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        if (misc[2]) {
          // y = ((0 + part_0) + part_1) + ...: four float4 of each split in flight per thread.
          const float4* pb0 = reinterpret_cast<const float4*>(a.partial + static_cast<size_t>(un.pbase) * (TC_NMAX * 256));
          const uint32_t nv = static_cast<uint32_t>(a.B) * 64u;   // float4 of the B columns' 256 rows
          constexpr uint32_t kT = TC_DEQ * 32;
          for (uint32_t v0 = static_cast<uint32_t>(tid); v0 < nv; v0 += 4u * kT) {
            float4 y[4];
#pragma unroll
            for (uint32_t k = 0; k < 4; ++k) y[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (uint32_t sp = 0; sp < un.nsplit; ++sp) {
              float4 t[4];
#pragma unroll
              for (uint32_t k = 0; k < 4; ++k) {
                const uint32_t v = v0 + k * kT;
                t[k] = v < nv ? __ldcg(pb0 + sp * (TC_NMAX * 64u) + v) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              }
#pragma unroll
              for (uint32_t k = 0; k < 4; ++k) {
                y[k].x += t[k].x;
                y[k].y += t[k].y;
                y[k].z += t[k].z;
                y[k].w += t[k].w;
              }
            }
#pragma unroll
            for (uint32_t k = 0; k < 4; ++k) {
              const uint32_t v = v0 + k * kT;
              if (v >= nv) break;
              const uint32_t bc = v >> 6, rr = 4u * (v & 63u);
              float* yr = a.Y + static_cast<int64_t>(bc) * a.N + r0 + rr;
              const float yv[4] = {y[k].x, y[k].y, y[k].z, y[k].w};
#pragma unroll
              for (uint32_t c = 0; c < 4; ++c)
                if (rr + c < rows) yr[c] = yv[c];
            }
          }
          if (tid == 0) a.counters[un.tile] = 0u;
        }
      }
    }
    if (!ok) abort_now();
  }

  __syncthreads();
  if (tid == 0 && misc[1]) atomicExch(a.err, kErrMmaTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 4 * TC_NMAX);
}

// The B tile of group column g (one CTA per g): Npad rows of 64 fp16 values
// x * sx in the K order of the A tiles, 128-byte swizzled; rows past B are zero.
__global__ void vbq_xprep_kernel(const uint16_t* __restrict__ X, int32_t K, int32_t B, int32_t Npad,
                                 const float* __restrict__ sx, uint8_t* __restrict__ bt) {
  const uint32_t g = blockIdx.x;
  grid_dep_launch();  // the dequant-MMA kernel may start its set-up
  grid_dep_wait();    // sx is complete
  for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(Npad) * 8u; i += blockDim.x) {
    const uint32_t bc = i >> 3, ch = i & 7u;
    uint4 pk = make_uint4(0u, 0u, 0u, 0u);
    if (bc < static_cast<uint32_t>(B)) {
      // Chunk ch holds codes 32 blk + s0 + t and those + 16 (t < 4), in pairs.
      const uint32_t* x32 = reinterpret_cast<const uint32_t*>(X + static_cast<int64_t>(bc) * K + g * GROUP +
                                                              32u * (ch >> 2) + 4u * (ch & 3u));  // 4-byte aligned
      const uint2 lo4 = make_uint2(x32[0], x32[1]), hi4 = make_uint2(x32[8], x32[9]);
      const float sxv = sx[bc];
      const float xa[4] = {bf16_lo(lo4.x), bf16_hi(lo4.x), bf16_lo(lo4.y), bf16_hi(lo4.y)};
      const float xb[4] = {bf16_lo(hi4.x), bf16_hi(hi4.x), bf16_lo(hi4.y), bf16_hi(hi4.y)};
      uint32_t ov[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        ov[t] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(xa[t] * sxv))) |
                (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(xb[t] * sxv))) << 16);
      pk = make_uint4(ov[0], ov[1], ov[2], ov[3]);
    }
    *reinterpret_cast<uint4*>(bt + static_cast<size_t>(g) * TC_BTILE + sw128(bc, ch)) = pk;
  }
}

// x scale per batch column: a power of two 2^p with max|x| * 2^p in [2^13, 2^14)
// (p limited to the float range).
__global__ void vbq_xscale_kernel(const uint16_t* __restrict__ X, int32_t K, float* __restrict__ sx) {
  __shared__ float red[32];
  grid_dep_launch();  // the B-tile kernel may start; it waits for this grid before reading sx
  const uint16_t* x = X + static_cast<int64_t>(blockIdx.x) * K;
  float m = 0.0f;
  for (int k = threadIdx.x; k < K; k += blockDim.x)
    m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[k]) << 16)));
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
    p = p > 127 ? 127 : (p < -126 ? -126 : p);
    sx[blockIdx.x] = ldexpf(1.0f, p);
  }
}

// Relative cost of one step of each class in the dequant, and of one pair's
// fixed work (its B tile, the MMA issue and the barriers).
constexpr double kTcStepCost[4] = {136.0, 170.0, 165.0, 140.0};
constexpr double kTcPairCost = 300.0;

struct TcState {
  void* mem = nullptr;
  const TcCta* ctas = nullptr;
  const TcUnit* units = nullptr;
  const TcPiece* pieces = nullptr;
  const uint32_t* pair_piece = nullptr;
  float* partial = nullptr;
  uint32_t* counters = nullptr;
  float* sx = nullptr;
  uint8_t* bt = nullptr;
  int32_t n_ctas = 0;
  bool built = false, eligible = false;
};

std::mutex g_tc_mu;
std::map<const vbq_matrix*, TcState> g_tc;

// Host plan: pieces of every (tile, group column) pair, then CTA ranges and units.
struct TcHost {
  std::vector<TcPiece> pieces;
  std::vector<uint32_t> pair_piece;
  std::vector<TcCta> ctas;
  std::vector<TcUnit> units;
  uint32_t n_blocks = 0;   // partial blocks
  bool ok = false;
};

TcHost build_tc_host(const vbq_matrix* m, int32_t sms) {
  TcHost H;
  const uint32_t G = static_cast<uint32_t>(m->G), nt = static_cast<uint32_t>(m->n_tiles);
  const uint64_t n_pairs = uint64_t(nt) * G;
  std::vector<double> cost(n_pairs, kTcPairCost);
  H.pair_piece.assign(n_pairs + 1, 0);
  for (uint32_t T = 0; T < nt; ++T) {
    const uint32_t st = T / SUPER, t = T % SUPER;
    for (uint32_t g = 0; g < G; ++g) {
      const uint64_t p = uint64_t(T) * G + g;
      H.pair_piece[p] = static_cast<uint32_t>(H.pieces.size());
      uint64_t bytes = 0;
      for (uint32_t r = m->block_run[size_t(st) * G + g]; r < m->block_run[size_t(st) * G + g + 1]; ++r) {
        const RunInfo& ri = m->runs[r];
        const RunHeader& h = ri.h;
        const uint32_t cs[4] = {0u, h.c1, h.c2, h.c3};
        const uint32_t lo = cs[t], hi = t + 1 < SUPER ? cs[t + 1] : h.n;
        if (lo >= hi) continue;
        const uint32_t ks = lo / 32, ke = (hi + 31) / 32, nsr = (h.n + 31u) / 32u;
        const uint64_t fb = full_step_bytes(h.cls);
        const uint64_t b0 = ri.off + HEADER_BYTES + ks * fb;
        const uint64_t b1 = ke == nsr ? ri.off + run_bytes(h.cls, h.n) : ri.off + HEADER_BYTES + ke * fb;
        TcPiece pc{};
        pc.off16 = static_cast<uint32_t>(b0 / 16);
        pc.bytes16 = static_cast<uint16_t>((b1 - b0) / 16);
        pc.cls = h.cls;
        pc.nst = static_cast<uint8_t>(ke - ks);
        pc.n = h.n;
        pc.ks = static_cast<uint16_t>(ks);
        pc.lo = static_cast<uint16_t>(lo);
        pc.hi = static_cast<uint16_t>(hi);
        if (b0 / 16 > UINT32_MAX) return H;
        H.pieces.push_back(pc);
        bytes += b1 - b0;
        cost[p] += (ke - ks) * kTcStepCost[h.cls];
      }
      if (bytes > uint64_t(TC_PIECE_BYTES)) return H;  // a pair must fit one stage
    }
  }
  H.pair_piece[n_pairs] = static_cast<uint32_t>(H.pieces.size());

  // CTA ranges: equal cost shares, each within the per-CTA limits (pairs, pieces, tiles).
  double total = 0.0;
  for (double c : cost) total += c;
  const double share = total / std::max<int32_t>(1, sms);
  std::vector<uint64_t> cuts{0};
  double acc = 0.0;
  uint64_t start = 0;
  for (uint64_t p = 0; p < n_pairs; ++p) {
    const uint64_t np = p + 1 - start;
    const uint32_t nq = H.pair_piece[p + 1] - H.pair_piece[start];
    const uint32_t ntl = static_cast<uint32_t>(p / G - start / G + 1);
    if (np > uint64_t(TC_MAX_PAIRS) || nq > uint32_t(TC_MAX_PIECES) || ntl > uint32_t(TC_MAX_UNITS)) {
      cuts.push_back(p);  // the range ends before p
      start = p;
    }
    acc += cost[p];
    if (acc >= share * static_cast<double>(cuts.size()) && p + 1 < n_pairs && start != p + 1) {
      cuts.push_back(p + 1);
      start = p + 1;
    }
  }
  if (cuts.back() != n_pairs) cuts.push_back(n_pairs);

  // Units, and each split tile's order of splits.
  std::vector<uint32_t> nsplit(nt, 0);
  for (size_t c = 0; c + 1 < cuts.size(); ++c) {
    TcCta ct{};
    ct.u0 = static_cast<uint32_t>(H.units.size());
    for (uint64_t p = cuts[c]; p < cuts[c + 1];) {
      const uint32_t T = static_cast<uint32_t>(p / G);
      const uint64_t pe = std::min<uint64_t>(cuts[c + 1], uint64_t(T + 1) * G);
      TcUnit u{};
      u.tile = T;
      u.p0 = static_cast<uint32_t>(p);
      u.p1 = static_cast<uint32_t>(pe);
      u.split = static_cast<uint16_t>(nsplit[T]++);
      H.units.push_back(u);
      p = pe;
    }
    ct.u1 = static_cast<uint32_t>(H.units.size());
    ct.q0 = H.pair_piece[cuts[c]];
    ct.q1 = H.pair_piece[cuts[c + 1]];
    if (ct.u1 > ct.u0) H.ctas.push_back(ct);
  }
  std::vector<uint32_t> pbase(nt, 0);
  for (uint32_t T = 0; T < nt; ++T)
    if (nsplit[T] > 1) {
      pbase[T] = H.n_blocks;
      H.n_blocks += nsplit[T];
    }
  for (TcUnit& u : H.units) {
    u.nsplit = static_cast<uint16_t>(nsplit[u.tile]);
    u.pbase = pbase[u.tile];
  }
  H.ok = true;
  return H;
}

// Builds (once) the matrix's tensor-core plan; false if the matrix is not eligible.
bool tc_state(const vbq_matrix* m, TcState** out, vbq_status* err) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  TcState& s = g_tc[m];
  *out = &s;
  *err = VBQ_OK;
  if (s.built) return s.eligible;
  s.built = true;
  if (!(m->max_scale <= TC_MAX_SCALE) || m->N <= 0 || m->K <= 0 || m->n_tiles <= 0) return false;
  const TcHost H = build_tc_host(m, gpu_info().sms);
  if (!H.ok || H.ctas.empty()) return false;
  auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t o_c = 0, o_u = o_c + al(sizeof(TcCta) * H.ctas.size());
  const size_t o_p = o_u + al(sizeof(TcUnit) * H.units.size());
  const size_t o_pp = o_p + al(sizeof(TcPiece) * std::max<size_t>(1, H.pieces.size()));
  const size_t o_cnt = o_pp + al(4 * H.pair_piece.size());
  const size_t o_sx = o_cnt + al(4 * static_cast<size_t>(m->n_tiles));
  const size_t o_bt = o_sx + al(4 * TC_NMAX);
  const size_t o_part = o_bt + al(static_cast<size_t>(m->G) * TC_BTILE);
  const size_t total = o_part + size_t(H.n_blocks) * TC_NMAX * 256 * 4;
  cudaError_t e = dev_alloc(&s.mem, total);
  char* b = static_cast<char*>(s.mem);
  if (e == cudaSuccess) e = cudaMemcpy(b + o_c, H.ctas.data(), sizeof(TcCta) * H.ctas.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(b + o_u, H.units.data(), sizeof(TcUnit) * H.units.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !H.pieces.empty())
    e = cudaMemcpy(b + o_p, H.pieces.data(), sizeof(TcPiece) * H.pieces.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(b + o_pp, H.pair_piece.data(), 4 * H.pair_piece.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(b + o_cnt, 0, 4 * static_cast<size_t>(m->n_tiles));
  if (e != cudaSuccess) {
    if (s.mem) cudaFree(s.mem);
    s.mem = nullptr;
    *err = cuda_fail(e, "vbq_gemm_smallbatch: tensor-core plan");
    s.built = false;
    return false;
  }
  s.ctas = reinterpret_cast<const TcCta*>(b + o_c);
  s.units = reinterpret_cast<const TcUnit*>(b + o_u);
  s.pieces = reinterpret_cast<const TcPiece*>(b + o_p);
  s.pair_piece = reinterpret_cast<const uint32_t*>(b + o_pp);
  s.counters = reinterpret_cast<uint32_t*>(b + o_cnt);
  s.sx = reinterpret_cast<float*>(b + o_sx);
  s.bt = reinterpret_cast<uint8_t*>(b + o_bt);
  s.partial = reinterpret_cast<float*>(b + o_part);
  s.n_ctas = static_cast<int32_t>(H.ctas.size());
  cudaFuncSetAttribute(vbq_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kBytes);
  s.eligible = true;
  return true;
}

}  // namespace

bool tc_eligible(const vbq_matrix* m) {
  TcState* s = nullptr;
  vbq_status err = VBQ_OK;
  return tc_state(m, &s, &err);
}

void tc_forget(const vbq_matrix* m) {
  std::lock_guard<std::mutex> lock(g_tc_mu);
  auto it = g_tc.find(m);
  if (it == g_tc.end()) return;
  if (it->second.mem) cudaFree(it->second.mem);
  g_tc.erase(it);
}

vbq_status launch_gemm_tc(const vbq_matrix* m, const uint16_t* X, int32_t B, float* Y, cudaStream_t st) {
  if (B < 1 || B > TC_NMAX) return fail(VBQ_ERR_INVALID_ARG, "tensor-core path: batch out of range");
  TcState* s = nullptr;
  vbq_status err = VBQ_OK;
  if (!tc_state(m, &s, &err)) return err != VBQ_OK ? err : fail(VBQ_ERR_UNSUPPORTED, "tensor-core path: not eligible");
  int* chk = device_check_word();
  if (!chk) return fail(VBQ_ERR_CUDA, "device check word");
  const int32_t npad = (B + 15) & ~15;
  note_launches(2);
  vbq_xscale_kernel<<<B, 256, 0, st>>>(X, static_cast<int32_t>(m->K), s->sx);
  VBQ_CUDA_TRY(cudaGetLastError());
  // The two kernels after the first are programmatic dependents: each starts
  // while the one before runs and waits for it (griddepcontrol.wait) before
  // reading its output.
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(m->G));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_xprep_kernel, X, static_cast<int32_t>(m->K), B, npad,
                                  static_cast<const float*>(s->sx), s->bt));
  TcArgs a{};
  a.data = m->data;
  a.ctas = s->ctas;
  a.units = s->units;
  a.pieces = s->pieces;
  a.pair_piece = s->pair_piece;
  a.partial = s->partial;
  a.counters = s->counters;
  a.bt = s->bt;
  a.sx = s->sx;
  a.Y = Y;
  a.B = B;
  a.Npad = npad;
  a.K = static_cast<int32_t>(m->K);
  a.G = m->G;
  a.N = m->N;
  a.err = chk;
  note_launches(1);
  cfg.gridDim = dim3(static_cast<unsigned>(s->n_ctas));
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = TcSmem::kBytes;
  VBQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, vbq_gemm_tc_kernel, a));
  return VBQ_OK;
}

}  // namespace vbq
