// Work plans for the GEMV kernels: which CTA and warp streams which bytes.
//
// A launch covers one or more packed matrices ("segments"). Their step records,
// tile after tile, form one byte stream. make_plan cuts that stream at step
// borders into n_ctas equal-byte CTA ranges, each range into units at tile
// borders, and each unit into SLICES equal-byte warp slices (layout.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "layout.h"

namespace vbq {

// Host copies of one packed matrix's side tables.
struct SegTables {
  const uint32_t* run_desc = nullptr;
  const uint32_t* run_off = nullptr;    // n_runs + 1 entries
  const uint32_t* tile_row0 = nullptr;  // n_tiles + 1 entries
  const uint32_t* tile_run0 = nullptr;  // n_tiles + 1 entries
  int32_t n_tiles = 0;
  int32_t n_runs = 0;
};

struct Plan {
  std::vector<UnitRec> units;     // n_ctas * umax slots
  std::vector<SliceRec> slices;   // SLICES per slot
  int32_t n_ctas = 0;
  int32_t umax = 0;               // unit slots per CTA
  uint64_t partial_rows = 0;      // rows of partial storage per batch column
  uint32_t n_counters = 0;
};

// Work model used to balance CTAs and warps: relative time per step of each
// bit class, per run, and per group column a warp has to prepare. Fitted to
// GEMV timings on a B300 (65536 x 4096 matrices of one class each, and the
// mixed allocation): a 1-bit step costs about 2.4 8-bit steps (it adds 32
// entries into the row accumulators, an 8-bit step 4), a run's set-up about
// 1.6 1-bit steps, and a column's lookup tables about 1.9.
constexpr uint32_t kCostStep[4] = {61, 47, 39, 25};
constexpr uint32_t kCostRun = 99;
constexpr uint32_t kCostColumn = 117;

// Number of CTAs for a launch over total_bytes: one per SM at most, but no
// fewer than 32 KB each, and never more than MAX_UNITS_PER_CTA units a CTA.
int32_t plan_ctas(uint64_t total_bytes, int sms);

// Builds the plan. If a CTA would get more than max_units units, the CTA count
// grows until none does. With whole_columns, every cut falls at the start of a
// (tile, group column), so each unit covers whole columns (the tensor-core
// path dequantizes one column of a tile at a time).
Plan make_plan(const std::vector<SegTables>& segs, int32_t n_ctas, int max_units, bool whole_columns = false);

// What each warp copies, in order: for CTA c and warp w of a W-warp CTA, the
// byte ranges of its slices of every unit (and, for a program of several
// launches, of every launch in turn). A piece is (address >> 4) << 20 | (bytes >> 4).
struct PieceSet {
  std::vector<uint64_t> pieces;
  std::vector<uint32_t> start;  // [n_ctas * W + 1]: first piece of each warp
  std::vector<uint32_t> bytes;  // [n_ctas * W]: bytes each warp copies
};
inline uint64_t make_piece(const uint8_t* addr, uint64_t bytes) {
  return ((reinterpret_cast<uint64_t>(addr) >> 4) << 20) | (bytes >> 4);
}
// Whether (addr, bytes) survives that encoding: 16-byte aligned, addr below
// 2^48 and bytes below 16 MiB.
inline bool piece_fits(const uint8_t* addr, uint64_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(addr);
  return (a & 15u) == 0 && (bytes & 15u) == 0 && a < (uint64_t(1) << 48) && bytes < (uint64_t(1) << 24);
}
// Appends, for each (CTA, warp), the pieces of plan p over segments whose data
// bases are seg_data. With W = 8 a warp takes the plan's slices 2w and 2w+1.
// Returns false if a piece does not fit the encoding (piece_fits).
bool append_pieces(const Plan& p, const std::vector<const uint8_t*>& seg_data, int W,
                   std::vector<std::vector<uint64_t>>* per_warp);
PieceSet finish_pieces(const std::vector<std::vector<uint64_t>>& per_warp);

// A plan's device copy: units, slices, arrival counters (zeroed) and partial
// rows for up to max_nb batch columns, plus the piece lists of the 16-warp and
// 8-warp kernels, in one allocation.
struct DevicePlan {
  void* base = nullptr;
  const UnitRec* units = nullptr;
  const SliceRec* slices = nullptr;
  uint32_t* counters = nullptr;
  float* partial = nullptr;
  const uint64_t* pieces16 = nullptr;
  const uint32_t* start16 = nullptr;
  const uint32_t* bytes16 = nullptr;
  const uint64_t* pieces8 = nullptr;
  const uint32_t* start8 = nullptr;
  const uint32_t* bytes8 = nullptr;
  int32_t n_ctas = 0;
  int32_t umax = 0;
  int64_t bytes = 0;
};

// Allocates and uploads (synchronously on stream). seg_data are the device
// bases of the plan's segments (for the piece lists). Returns cudaSuccess or the error.
cudaError_t upload_plan(const Plan& p, int max_nb, const std::vector<const uint8_t*>& seg_data,
                        cudaStream_t stream, DevicePlan* out);
void free_plan(DevicePlan* p);

}  // namespace vbq
