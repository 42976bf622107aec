// mx_quant.cuh - the MXFP8 quantisation step of the standalone quantize
// kernel (one lane per 32-element block) and of the fused small-M GEMM (four
// lanes per block): the same decisions on the same bf16 bits, so both produce
// the same bytes.
//
// Rule (OCP MX v1.0, section 6.3, for the "MXFP8 format" of the
// CompressedTensorsW8A8Mxfp8 page): per 32-element block, e = floor(log2 amax)
// - 8 clamped to [-127, 127], scale byte e + 127, element E4M3(x / 2^e) with
// round-to-nearest-even and saturation to +-448; a block holding Inf/NaN gets
// byte 0xFF and elements 0x7F.  Decided on bf16 bit patterns:
//   * |x| as an integer is (bits & 0x7FFF): integer order is value order for
//     non-negative floats, and Inf/NaN are exactly the patterns >= 0x7F80;
//   * for a finite amax with exponent field E, floor(log2 amax) = E - 127, so
//     the byte is max(E - 8, 0) (zero and subnormal blocks clamp to 0);
//   * 2^-e = 2^(127 - byte) is a normal fp32 for byte in [0, 246], and x * 2^-e
//     is exact in fp32 unless it underflows, which rounds to a signed zero in
//     E4M3 either way;
//   * fp32 -> E4M3 is the hardware's cvt.rn.satfinite.e4m3x2.
#pragma once

#include <stdint.h>

#include "mx_ptx.cuh"

namespace mx {

// Quantise 8 consecutive bf16 values (one 16-byte load) that are one quarter
// of a 32-element block; the block's four quarters sit in four consecutive
// lanes (lane % 4 = quarter).  Must be called by all 32 lanes of the warp.
// Returns the block's scale byte (same in the four lanes) and the 8 codes.
__device__ __forceinline__ uint32_t quantize_quarter_block(const uint4 v, uint2& codes) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  // |x| of both halves at once; unsigned 16-bit max per half
  uint32_t m2 = __vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
  uint32_t amax = max(m2 & 0xFFFFu, m2 >> 16);
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));

  const bool nonfinite = amax >= 0x7F80u;
  const uint32_t E = amax >> 7;
  const uint32_t sbyte = nonfinite ? 0xFFu : (E > 8u ? E - 8u : 0u);
  const float mul = __uint_as_float((254u - (nonfinite ? 0u : sbyte)) << 23);

  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * mul;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * mul;
    c[i] = cvt_e4m3x2(lo, hi);
  }
  codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  if (nonfinite) codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  return sbyte;
}

// One bf16 value per lane, the 32 lanes of the warp one 32-element block (lane
// i = element i): the same decisions as quantize_block32 on the same bits.
// Must be called by all 32 lanes.  Returns this lane's E4M3 code; the block's
// scale byte goes to *sbyte (the same in every lane).
__device__ __forceinline__ uint32_t quantize_lane_block(uint32_t bf16_bits, uint32_t* sbyte) {
  const uint32_t amax = __reduce_max_sync(0xFFFFFFFFu, bf16_bits & 0x7FFFu);
  const bool nonfinite = amax >= 0x7F80u;
  const uint32_t E = amax >> 7;
  const uint32_t sb = nonfinite ? 0xFFu : (E > 8u ? E - 8u : 0u);
  const float mul = __uint_as_float((254u - (nonfinite ? 0u : sb)) << 23);
  const uint32_t code = cvt_e4m3x2(__uint_as_float(bf16_bits << 16) * mul, 0.f) & 0xFFu;
  *sbyte = sb;
  return nonfinite ? 0x7Fu : code;
}

// Element formats of a quantised block: kFmtE4M3 for activations and MXFP8
// weights; kFmtE2M3 / kFmtE3M2 for MXFP6 weights (the mxfp6 page's
// kMxfp6E2M3Static / kMxfp6E3M2Static), one 6-bit code per byte here.
constexpr int kFmtE4M3 = 0;
constexpr int kFmtE2M3 = 1;
constexpr int kFmtE3M2 = 2;

// emax of the element format: floor(log2 of its largest finite value).
__host__ __device__ constexpr uint32_t fmt_emax(int fmt) { return fmt == kFmtE2M3 ? 2u : (fmt == kFmtE3M2 ? 4u : 8u); }

template <int FMT>
__device__ __forceinline__ uint32_t cvt_fmt_x2(float lo, float hi) {
  if (FMT == kFmtE2M3) return cvt_e2m3x2(lo, hi);
  if (FMT == kFmtE3M2) return cvt_e3m2x2(lo, hi);
  return cvt_e4m3x2(lo, hi);
}

// One whole 32-element block per lane: 16 bf16 words in, 32 codes (two
// 16-byte words) and the scale byte out.  The same decisions as
// quantize_quarter_block, without cross-lane shuffles: a warp quantises 32
// blocks with ~3x fewer instructions per element.  FMT != kFmtE4M3 quantises
// to an FP6 element instead (scale byte max(E - emax, 0) with that format's
// emax; a block holding Inf/NaN gets byte 0xFF and codes 0x00, since FP6 has
// no NaN code).
template <int FMT = kFmtE4M3>
__device__ __forceinline__ uint32_t quantize_block32(const uint4 (&v)[4], uint4& c0, uint4& c1) {
  uint32_t w[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[4 * q] = v[q].x;
    w[4 * q + 1] = v[q].y;
    w[4 * q + 2] = v[q].z;
    w[4 * q + 3] = v[q].w;
  }
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = __vmaxu2(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __vmaxu2(m[i], m[i + 4]);
  m[0] = __vmaxu2(__vmaxu2(m[0], m[2]), __vmaxu2(m[1], m[3]));
  const uint32_t amax = max(m[0] & 0xFFFFu, m[0] >> 16);
  const bool nonfinite = amax >= 0x7F80u;
  const uint32_t E = amax >> 7;
  constexpr uint32_t kEmax = fmt_emax(FMT);
  const uint32_t sbyte = nonfinite ? 0xFFu : (E > kEmax ? E - kEmax : 0u);
  const float mul = __uint_as_float((254u - (nonfinite ? 0u : sbyte)) << 23);
  constexpr uint32_t kNanCodes = FMT == kFmtE4M3 ? 0x7F7F7F7Fu : 0u;
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = cvt_fmt_x2<FMT>(__uint_as_float(w[2 * i] << 16) * mul,
                                       __uint_as_float(w[2 * i] & 0xFFFF0000u) * mul);
    const uint32_t bb = cvt_fmt_x2<FMT>(__uint_as_float(w[2 * i + 1] << 16) * mul,
                                        __uint_as_float(w[2 * i + 1] & 0xFFFF0000u) * mul);
    o[i] = nonfinite ? kNanCodes : (a | (bb << 16));
  }
  c0 = make_uint4(o[0], o[1], o[2], o[3]);
  c1 = make_uint4(o[4], o[5], o[6], o[7]);
  return sbyte;
}

}  // namespace mx
