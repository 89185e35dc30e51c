// Packed VBQ layout: one definition shared by the host packer, the planner and the kernels.
//
// The pages ("Variable Bit-width Quantization ...", abstract) state only that a
// fixed per-group bit allocation can be stored as packed low-bit codes; they
// give no format. Everything below is this library's own design for sm_103a.
//
// Rows are cut into tiles of at most TILE_MAX rows. Tiles are cut where the
// running byte count reaches a target, so tiles carry about equal bytes. Within
// a tile, the entries (one entry = the 64 codes of one (row, g) group) are
// ordered by group column g, then by bit-class (1, 2, 4, 8), then by row. All
// entries of one (tile, g, class) form a "run". A run is stored as a sequence
// of "steps" of up to 32/b entries each, so that every lane of a warp reads
// exactly 8 code bytes of a step: lane i holds slice (i % b) of entry (i / b).
// Every step of a run is full except possibly the last one. A step's record is
//
//     [codes: e*8*b bytes][scales: e * fp16][rows: e * u8 row-in-tile][pad to 16 B]
//
// Within an entry of 1, 2 or 4 bits, the codes are stored as bit-planes: plane
// p (bit p of every code) fills bytes [8p, 8p+8) with code m's bit at bit m,
// little-endian. Lane slice s of such an entry is therefore plane s. Since
// q - (2^b - 1)/2 = sum_p 2^p (q_p - 1/2), every plane is decoded like a 1-bit
// group and the planes are combined with weights 2^p. An 8-bit entry stores
// code m in byte m, so its lane slice s holds codes [8s, 8s+8).
//
// Side tables, all uint32:
//     run_desc[n_runs]       g | cls << 16 | (n-1) << 18     (cls = log2 b, n = entries)
//     run_off[n_runs+1]      first record of the run, in 16-byte units from the data base
//     tile_row0[n_tiles+1]   first row of each tile (tile_row0[n_tiles] = N)
//     tile_run0[n_tiles+1]   first run of each tile
#pragma once

#include <stdint.h>

#if !defined(__CUDACC__) && !defined(__host__)
#define __host__
#endif
#if !defined(__CUDACC__) && !defined(__device__)
#define __device__
#endif

namespace vbq {

constexpr int GROUP = 64;
constexpr int TILE_MAX = 256;      // a row index in a tile fits one byte
constexpr int STEP_LANES = 32;
constexpr int LOG_STEP_LANES = 5;
constexpr int LANE_BYTES = 8;      // code bytes per lane per step
constexpr int MAX_G = 65535;       // group column fits 16 bits

__host__ __device__ inline constexpr int cls_bits(int cls) { return 1 << cls; }
__host__ __device__ inline constexpr uint32_t entries_per_step(uint32_t cls) { return STEP_LANES >> cls; }

__host__ __device__ inline uint32_t make_run(uint32_t g, uint32_t cls, uint32_t n) {
  return g | (cls << 16) | ((n - 1u) << 18);
}
__host__ __device__ inline uint32_t run_g(uint32_t d) { return d & 0xFFFFu; }
__host__ __device__ inline uint32_t run_cls(uint32_t d) { return (d >> 16) & 3u; }
__host__ __device__ inline uint32_t run_n(uint32_t d) { return ((d >> 18) & 255u) + 1u; }
__host__ __device__ inline uint32_t run_steps(uint32_t d) {
  const uint32_t eps = entries_per_step(run_cls(d));
  return (run_n(d) + eps - 1u) / eps;
}

// Byte layout of a step record with e entries of class cls.
__host__ __device__ inline constexpr uint32_t rec_code_bytes(uint32_t cls, uint32_t e) { return e * 8u << cls; }
__host__ __device__ inline constexpr uint32_t rec_scale_off(uint32_t cls, uint32_t e) { return rec_code_bytes(cls, e); }
__host__ __device__ inline constexpr uint32_t rec_row_off(uint32_t cls, uint32_t e) { return rec_code_bytes(cls, e) + 2u * e; }
__host__ __device__ inline constexpr uint32_t rec_bytes(uint32_t cls, uint32_t e) {
  return (rec_code_bytes(cls, e) + 3u * e + 15u) & ~15u;
}
// Bytes of a full step of class cls.
__host__ __device__ inline constexpr uint32_t full_step_bytes(uint32_t cls) { return rec_bytes(cls, entries_per_step(cls)); }

// ---- work plan (built on the host, read by the GEMV kernels) ----
//
// A plan gives each CTA one contiguous byte range of the packed stream of one
// launch (the concatenation of the launch's matrices, tile after tile). The
// part of a CTA's range that falls in one tile is a "unit". A tile cut between
// CTAs has nsplit > 1 units; each writes a partial row sum and the last one to
// finish adds them in split order. Each unit is further cut into SLICES
// equal-byte slices, one per warp. CTA c owns the unit slots
// [c*umax, (c+1)*umax); its units come first, and an empty slot has nsplit 0.
constexpr int SLICES = 16;
constexpr int MAX_UNITS_PER_CTA = 32;  // one unit per lane of a warp

struct UnitRec {           // 32 bytes
  uint32_t seg;            // matrix of the launch
  uint32_t tile;           // tile within that matrix
  uint32_t split, nsplit;  // this unit's index among the units of its tile, and their count (0: empty slot)
  uint32_t pbase;          // split tiles: first partial row (times the batch width at run time)
  uint32_t cnt;            // split tiles: arrival counter index
  uint32_t r0, rows;       // the tile's first row and row count
};

struct SliceRec {          // 32 bytes
  uint32_t run0, k0;       // first step: step k0 of run run0
  uint32_t run1, k1;       // end (exclusive): step k1 of run run1 (k1 = 0: the end of run run1 - 1)
  uint32_t b0, b1;         // byte range of the slice's records, in 16-byte units
  uint32_t g0;             // group column of the first run (0 for an empty slice)
  uint32_t pad;
};

}  // namespace vbq
