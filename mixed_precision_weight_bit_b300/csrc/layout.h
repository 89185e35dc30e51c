// Packed VBQ layout: one definition shared by the host packer and the kernels.
//
// The pages ("Variable Bit-width Quantization ...", abstract) say only that the
// per-group allocation "maps directly to packed low-bit storage". Everything
// below is this library's own design for sm_103a.
//
// Rows are cut into tiles of at most TILE_MAX rows. Tiles are cut where the
// running byte count reaches a target, so tiles carry about equal bytes. A
// tile's data is a stream of "steps", ordered by group column g, then by
// bit-class (1, 2, 4, 8), then by row. Each step covers up to 32/b entries
// (one entry = the 64 codes of one (row, g) group) of a single class b. Its
// codes fill at most 256 bytes, so that every lane of a warp reads exactly 8
// code bytes: lane i holds slice (i % b) of entry (i / b). A step's record is
//
//     [codes: e*8*b bytes][scales: e * fp16][rows: e * u8 row-in-tile][pad to 16 B]
//
// Within an entry, code m of the group sits at bits [m*b, m*b + b) of the
// entry's 8*b bytes, read as one little-endian integer. Lane slice s of a
// class-b entry therefore holds codes [s*64/b, (s+1)*64/b) in its 8 bytes.
//
// Side tables, all uint32:
//     step_desc[n_steps]     g | cls << 16 | (e-1) << 18     (cls = log2 b)
//     step_off[n_steps+1]    record start in 16-byte units from the data base
//     tile_row0[n_tiles+1]   first row of each tile (tile_row0[n_tiles] = N)
//     tile_step0[n_tiles+1]  first step of each tile
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
constexpr int LANE_BYTES = 8;      // code bytes per lane per step
constexpr int MAX_G = 65535;       // group column fits 16 bits

__host__ __device__ inline constexpr int cls_bits(int cls) { return 1 << cls; }
__host__ __device__ inline constexpr int entries_per_step(int cls) { return STEP_LANES >> cls; }

__host__ __device__ inline uint32_t make_desc(uint32_t g, uint32_t cls, uint32_t e) {
  return g | (cls << 16) | ((e - 1u) << 18);
}
__host__ __device__ inline uint32_t desc_g(uint32_t d) { return d & 0xFFFFu; }
__host__ __device__ inline uint32_t desc_cls(uint32_t d) { return (d >> 16) & 3u; }
__host__ __device__ inline uint32_t desc_e(uint32_t d) { return ((d >> 18) & 31u) + 1u; }

// Byte layout of a step record with e entries of class cls.
__host__ __device__ inline uint32_t rec_code_bytes(uint32_t cls, uint32_t e) { return e * 8u << cls; }
__host__ __device__ inline uint32_t rec_scale_off(uint32_t cls, uint32_t e) { return rec_code_bytes(cls, e); }
__host__ __device__ inline uint32_t rec_row_off(uint32_t cls, uint32_t e) { return rec_code_bytes(cls, e) + 2u * e; }
__host__ __device__ inline uint32_t rec_bytes(uint32_t cls, uint32_t e) {
  return (rec_code_bytes(cls, e) + 3u * e + 15u) & ~15u;
}

}  // namespace vbq
