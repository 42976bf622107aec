// mx_layout.cuh - byte layout of the packed scale factors.
//
// The tensor cores read block scales from tensor memory; tcgen05.cp fills
// tensor memory from 512-byte shared-memory "atoms".  An atom holds the E8M0
// scales of 128 rows x 4 consecutive 32-element blocks along K (one 128-wide
// K tile).  Within an atom, row r (0..127) and block j (0..3) sit at
//     (r % 32) * 16 + (r / 32) * 4 + j
// so each 16-byte line carries rows {i, i+32, i+64, i+96}.
//
// Atoms are stored K-tile major, then row-tile:
//     atom(b, kt, rt) = (b * KT + kt) * RT + rt,   RT = ceil(R / 128),
//                                                  KT = ceil(K / 128)
// so the atoms of consecutive 128-row tiles at one K tile are adjacent, and a
// 256-row operand tile reads 1 KB contiguous per K tile.  Rows >= R and blocks
// >= K/32 are padding.  The scale repack (sf_pack_kernel) writes them as 0;
// the quantise kernel writing packed scales leaves them as they were, which
// only affects accumulator rows >= R, and those are never stored.
#pragma once

#include <stdint.h>

namespace mx {

constexpr int kAtomRows = 128;
constexpr int kAtomBlocks = 4;
constexpr int kAtomBytes = 512;
constexpr int kTileK = 128;  // K elements covered by one atom column group

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__host__ __device__ __forceinline__ int64_t sf_packed_bytes(int64_t B, int64_t R, int64_t K) {
  return B * ceil_div(K, kTileK) * ceil_div(R, kAtomRows) * kAtomBytes;
}

// Bytes one TMA copy of a `rows` x 128-element weight tile counts on its
// mbarrier: the global bytes it reads, 128 per row for E4M3 and 96 per row
// for packed 6-bit FP6 codes (wfmt != 0; expanded to 128 bytes per row in
// shared memory, the same tile shape as E4M3).
__host__ __device__ __forceinline__ uint32_t weight_tile_tx_bytes(int rows, int wfmt) {
  return static_cast<uint32_t>(rows) * (wfmt == 0 ? 128u : 96u);
}

// Offset of the scale of (batch b, row r, block kb) inside the packed buffer.
__host__ __device__ __forceinline__ int64_t sf_packed_offset(int64_t b, int64_t r, int64_t kb,
                                                            int64_t RT, int64_t KT) {
  const int64_t kt = kb >> 2, j = kb & 3;
  const int64_t rt = r >> 7, rr = r & 127;
  return ((b * KT + kt) * RT + rt) * kAtomBytes + (rr & 31) * 16 + (rr >> 5) * 4 + j;
}

}  // namespace mx
