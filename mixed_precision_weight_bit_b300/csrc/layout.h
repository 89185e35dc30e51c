// Packed VBQ layout: one definition shared by the host packer, the planner and the kernels.
//
// The pages ("Variable Bit-width Quantization ...", abstract) state only that a
// fixed per-group bit allocation can be stored as packed low-bit codes; they
// give no format. Everything below is this library's own design for sm_103a.
//
// Rows are cut into tiles of TILE = 256 rows (a row index inside a tile fits
// one byte) and tiles into super-tiles of SUPER = 4 tiles (1024 rows); the
// last ones may be shorter. The packed stream of a matrix is a sequence of
// RUN records in this order: super-tile, then group column g, then bit class
// (1, 2, 4, 8 bits). A run holds every group of one (super-tile, g) with that
// bit-width, ordered by row; empty runs are left out. A run is
//
//     [16-byte RunHeader][step][step]...
//
// and a step holds up to 32 groups ("entries"); lane l of a warp works on
// entry l. A step record of class c (b = 2^c bits) with e entries is
//
//     [codes: e * 8 * b bytes][scales: e * fp16][rows: e * u8 row-in-tile][pad to 16 B]
//
// Every step of a run is full (32 entries) except possibly the last one. The
// tile of entry i of a run (counted from the run's start) is the number of
// prefix counts c1, c2, c3 of the header that are <= i.
//
// Codes of an entry (64 codes, 8*b bytes) are 2*b 32-bit words; word w holds
// codes [w*32/b, (w+1)*32/b).
//  * b = 1: the entry's 8 bytes sit at 8*j in the record (entry j); code m of
//    a word at bit m (little-endian bits).
//  * b = 2, 4, 8: the words go in 16-byte chunks of four, chunk q of entry j at
//    byte 16 * (q * e + j), so that the 32 lanes read one chunk each with no
//    bank conflict. Code r of a word (0 <= r < 32/b) sits in byte (r & 3) at
//    bit offset b * (r >> 2); then (word >> (b*i)) & mask puts codes
//    4i .. 4i+3 into the four bytes of a word, ready for a byte dot product.
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
constexpr int TILE = 256;          // rows per tile; a row index in a tile fits one byte
constexpr int SUPER = 4;           // tiles per super-tile
constexpr int SROWS = TILE * SUPER;  // rows per super-tile
constexpr int STEP_LANES = 32;     // entries per full step
constexpr int MAX_G = 65535;       // group columns per matrix (g fits 16 bits)
constexpr int HEADER_BYTES = 16;

__host__ __device__ inline constexpr int cls_bits(int cls) { return 1 << cls; }
__host__ __device__ inline constexpr uint32_t entries_per_step(uint32_t) { return STEP_LANES; }

// Byte layout of a step record with e entries of class cls.
__host__ __device__ inline constexpr uint32_t rec_code_bytes(uint32_t cls, uint32_t e) { return e * 8u << cls; }
__host__ __device__ inline constexpr uint32_t rec_scale_off(uint32_t cls, uint32_t e) { return rec_code_bytes(cls, e); }
__host__ __device__ inline constexpr uint32_t rec_row_off(uint32_t cls, uint32_t e) {
  return rec_code_bytes(cls, e) + 2u * e;
}
__host__ __device__ inline constexpr uint32_t rec_bytes(uint32_t cls, uint32_t e) {
  return (rec_code_bytes(cls, e) + 3u * e + 15u) & ~15u;
}
// Bytes of a full step of class cls.
__host__ __device__ inline constexpr uint32_t full_step_bytes(uint32_t cls) { return rec_bytes(cls, entries_per_step(cls)); }
// Steps of a run of n entries, and its bytes including the header.
__host__ __device__ inline constexpr uint32_t run_steps(uint32_t, uint32_t n) { return (n + STEP_LANES - 1u) >> 5; }
__host__ __device__ inline constexpr uint32_t run_bytes(uint32_t cls, uint32_t n) {
  return HEADER_BYTES + (n / entries_per_step(cls)) * full_step_bytes(cls) +
         ((n % entries_per_step(cls)) ? rec_bytes(cls, n % entries_per_step(cls)) : 0u);
}

struct RunHeader {   // 16 bytes, at the start of every run
  uint32_t row0;     // first row of the run's super-tile
  uint16_t g;        // group column
  uint8_t cls;       // log2 of the bit-width
  uint8_t ntl;       // tiles in the super-tile (1 .. SUPER)
  uint16_t n;        // entries (1 .. SROWS)
  uint16_t c1, c2, c3;  // entries in the run's tiles before tile 1, 2 and 3 (n if the tile does not exist)
};
static_assert(sizeof(RunHeader) == HEADER_BYTES, "run header is 16 bytes");

// Tile (0 .. SUPER-1) inside the super-tile of entry i of a run.
__host__ __device__ inline uint32_t entry_tile(const RunHeader& h, uint32_t i) {
  return static_cast<uint32_t>(i >= h.c1) + static_cast<uint32_t>(i >= h.c2) + static_cast<uint32_t>(i >= h.c3);
}

// Byte offset of code word w (0 <= w < 2b) of entry j in a step record of class cls with e entries.
__host__ __device__ inline constexpr uint32_t code_word_off(uint32_t cls, uint32_t e, uint32_t j, uint32_t w) {
  return cls == 0 ? 8u * j + 4u * w : ((w >> 2) * e + j) * 16u + 4u * (w & 3u);
}

// Bit offset of code r (0 <= r < 32/b) inside its 32-bit word, b >= 2.
__host__ __device__ inline constexpr uint32_t code_bit(uint32_t b, uint32_t r) { return (r & 3u) * 8u + b * (r >> 2); }

}  // namespace vbq
