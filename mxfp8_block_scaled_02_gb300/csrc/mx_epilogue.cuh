// mx_epilogue.cuh - the GEMM epilogue's MXFP8 hand-off: quantise the bf16
// output for the next layer inside the epilogue (the QuantizedActivation
// hand-off of "AiterFlyDSLMxfp8LinearKernel.apply_weights", aiter_flydsl page,
// where the previous op passes its output already quantised; here the
// producing GEMM does the quantisation while the values are in registers).
//
// An epilogue thread holds one output row, 128 consecutive columns starting at
// a multiple of 128, as 64 bf16x2 words (word w = columns 2w, 2w + 1): exactly
// four 32-element MX blocks along the next layer's K, and in the packed scale
// layout (mx_layout.cuh) the four scale bytes of one row of one atom, one
// aligned 32-bit word.  The bytes are those of the standalone quantiser
// (quantize_block32 on the same bf16 bits).
#pragma once

#include <stdint.h>

#include "mx_layout.cuh"
#include "mx_quant.cuh"

namespace mx {

// Codes go to yq[b][row][n0 .. n0 + 127] ([B, M, N] E4M3, row-major) and the
// scale word to the packed atoms of (B, M, N): RTY = ceil(M / 128) row tiles,
// KTY = N / 128 K tiles.  Rows >= M are not stored; N % 128 == 0 (the caller
// checks), so the four blocks are all inside the row when n0 < N.
__device__ __forceinline__ void store_quantized_row128(const uint32_t (&packed)[64], uint8_t* __restrict__ yq,
                                                       uint8_t* __restrict__ ysf, int b, int row, int n0, int M,
                                                       int N, int RTY, int KTY) {
  if (row >= M || n0 >= N) return;
  uint8_t* q = yq + (static_cast<int64_t>(b) * M + row) * N + n0;
  uint32_t sword = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 v[4] = {make_uint4(packed[16 * c], packed[16 * c + 1], packed[16 * c + 2], packed[16 * c + 3]),
                        make_uint4(packed[16 * c + 4], packed[16 * c + 5], packed[16 * c + 6], packed[16 * c + 7]),
                        make_uint4(packed[16 * c + 8], packed[16 * c + 9], packed[16 * c + 10], packed[16 * c + 11]),
                        make_uint4(packed[16 * c + 12], packed[16 * c + 13], packed[16 * c + 14],
                                   packed[16 * c + 15])};
    uint4 c0, c1;
    sword |= quantize_block32(v, c0, c1) << (8 * c);
    reinterpret_cast<uint4*>(q + 32 * c)[0] = c0;
    reinterpret_cast<uint4*>(q + 32 * c)[1] = c1;
  }
  const int64_t atom = (static_cast<int64_t>(b) * KTY + n0 / kTileK) * RTY + (row >> 7);
  *reinterpret_cast<uint32_t*>(ysf + atom * kAtomBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4) = sword;
}

}  // namespace mx
