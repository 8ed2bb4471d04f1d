// layout.cuh -- shared-memory operand layouts of the tensor-core tiles.
//
// Every operand tile is built from 128-byte-swizzled "atoms": 8 rows of 128
// bytes (64 sixteen-bit elements per row); inside an atom the 16-byte chunk
// c of row r sits at chunk position (c XOR r).  An atom column covers 64
// elements along a row; a tile of R rows stores its atom columns one after
// another, each R/8 atoms (R * 128 bytes) long.
//
//   K-major use (contraction along the row):  start advances 32 bytes per
//     16-element step inside an atom column, stride between 8-row groups
//     (SBO) = 1024 bytes.
//   MN-major use (contraction across rows):   start advances 2048 bytes per
//     16-row step, SBO = 1024 bytes, LBO = bytes of one atom column.
#pragma once
#include <cstdint>

namespace gmm {

constexpr int kBN = 128;          // points per tile (tensor-core M of the logit contraction)
constexpr int kSlice = 128;       // components per CTA
constexpr int kAtomElems = 64;    // 16-bit elements per swizzled row
constexpr int kChunkBytes = 128 * 128;  // one atom column of a 128-row tile
constexpr int kRSlotBytes = 32 * 128;   // one R slot: 32 points x 64 components x 16 bit

// Byte offset of the 16-byte chunk `c16` (0..7) of row `r` inside one atom column.
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c16) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((c16 ^ (r & 7u)) << 4);
}

// The logit constant enters the logit contraction as one more 16-wide K step:
// an operand of 128 rows x 16 columns without swizzling (8-row x 16-byte core
// matrices; the two core matrices of a row group sit 128 bytes apart along K,
// row groups 256 bytes apart).  The data side of that step is the same in
// every row: 2^15, 2^4, 2^-7 in columns 0..2 and zeros elsewhere; the
// parameter side holds, per component, the constant split into three fp16
// pieces scaled by 2^-15, 2^-4 and 2^7, so that the products add up to it.
constexpr int kConstBytes = 128 * 16 * 2;   // 4 KB
constexpr uint32_t kConstLbo = 128;
constexpr uint32_t kConstSbo = 256;
__host__ __device__ constexpr int const_exp(int i) { return i == 0 ? 15 : i == 1 ? 4 : -7; }

// Byte offset of element (row, k) of a 128 x 16 operand in that layout.
__host__ __device__ __forceinline__ uint32_t const_off(uint32_t row, uint32_t k) {
  return (row >> 3) * kConstSbo + (k >> 3) * kConstLbo + (row & 7u) * 16u + (k & 7u) * 2u;
}

}  // namespace gmm
