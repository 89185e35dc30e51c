// Work plans for the batch-1 kernels: which CTA and warp handles which steps.
//
// An "item" is one GEMV over one or more packed matrices ("segments") that
// share an input vector (for example q, k and v). Its stream is the
// concatenation of the segments' run records (layout.h). The planner cuts the
// stream at step borders into one range per CTA and each CTA range into one
// range per warp, balancing a cost model. A CTA range may touch at most
// SLOTS_MAX consecutive super-tiles of the item (its shared-memory row
// accumulators) and at most CCAP group columns (its staged input).
//
// Item rows: segment s occupies item super-tiles [st_off[s], st_off[s] + n_super(s)),
// so item row = 1024 * st_off[s] + row in the matrix. Outputs are kept in this
// padded item-row space.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "layout.h"

namespace vbq {

#ifndef VBQ_KW
#define VBQ_KW 16
#endif
constexpr int KW = VBQ_KW;     // consumer warps per CTA of the batch-1 kernels
constexpr int SLOTS_MAX = 2;   // super-tiles a CTA range may touch
constexpr int CCAP = 64;       // group columns a CTA range may touch
constexpr int MAX_SEG = 3;     // segments per item

// Host copy of one run of a packed matrix.
struct RunInfo {
  uint64_t off;   // byte offset of the run header from the matrix data
  RunHeader h;    // the header as stored
  uint32_t st() const { return h.row0 / SROWS; }
};

// A warp's work inside one segment: steps [k0, k0 + nsteps) of the stream,
// counted from the run whose header is `first`.
struct SubRange {          // 32 bytes
  RunHeader first;         // header of the run the sub-range starts in
  uint32_t seg;            // segment of the item
  uint32_t k0;             // first step in that run; 0 means the range starts at the header
  uint32_t nsteps;         // steps in the sub-range (0: empty)
  uint32_t bytes;          // bytes the warp streams for it
};

struct WarpPlan {          // 128 bytes
  SubRange sub[MAX_SEG];
  uint32_t nsub;
  uint32_t pad[7];
};

// Columns a CTA stages: [a0, a1) then [b0, b1), packed into slots 0 .. n_cols-1.
struct CtaPlan {           // 32 bytes
  uint32_t st_base;        // first item super-tile the CTA touches
  uint32_t n_slots;        // item super-tiles it touches (<= SLOTS_MAX; 0 for an idle CTA)
  uint32_t a0, a1, b0, b1;
  uint32_t expect[SLOTS_MAX];  // per slot: CTAs that touch that super-tile (its arrivals)
};

__host__ __device__ inline uint32_t col_slot(const CtaPlan& c, uint32_t g) {
  return (g >= c.a0 && g < c.a1) ? g - c.a0 : (c.a1 - c.a0) + g - c.b0;
}

// Cost model of a warp's work: per step of each class, per run and per group
// column the warp prepares (lookup tables and fixed-point x).
constexpr double kCostStep[4] = {64.0, 81.0, 78.0, 64.0};
constexpr double kCostRun = 40.0;
constexpr double kCostColumn = 60.0;

struct SegPlanInput {
  const std::vector<RunInfo>* runs;
  const uint8_t* data;      // device base of the segment's records
  uint32_t n_super;
  uint32_t G;
};

struct ItemPlan {
  std::vector<WarpPlan> warps;   // n_ctas * KW
  std::vector<CtaPlan> ctas;     // n_ctas
  std::vector<uint32_t> arrivals;  // per item super-tile: CTAs that touch it
  std::vector<uint32_t> st_off;    // per segment: first item super-tile
  std::vector<uint64_t> sub_b0;    // per (warp, sub-range): first byte, from the segment's data
  uint32_t n_item_super = 0;
  int32_t n_ctas = 0;
  double total_cost = 0.0;
};

// Cuts the item into n_ctas * KW warp ranges. Returns false (with *why set) if
// the CTA ranges cannot respect SLOTS_MAX and CCAP with n_ctas CTAs.
bool make_item_plan(const std::vector<SegPlanInput>& segs, int32_t n_ctas, ItemPlan* out, const char** why);

// Appends, for each (CTA, warp), the byte pieces the warp streams for this
// item, in order. A piece is (address >> 4) << 20 | (bytes >> 4).
bool append_pieces(const ItemPlan& p, const std::vector<SegPlanInput>& segs,
                   std::vector<std::vector<uint64_t>>* per_warp);
inline uint64_t make_piece(const uint8_t* addr, uint64_t bytes) {
  return ((reinterpret_cast<uint64_t>(addr) >> 4) << 20) | (bytes >> 4);
}
inline bool piece_fits(const uint8_t* addr, uint64_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(addr);
  return (a & 15u) == 0 && (bytes & 15u) == 0 && a < (uint64_t(1) << 48) && bytes < (uint64_t(1) << 24);
}

struct PieceSet {
  std::vector<uint64_t> pieces;
  std::vector<uint32_t> start;  // [n_warps + 1]
  std::vector<uint32_t> bytes;  // [n_warps]
};
PieceSet finish_pieces(const std::vector<std::vector<uint64_t>>& per_warp);

}  // namespace vbq
