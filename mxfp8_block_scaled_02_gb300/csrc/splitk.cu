// splitk.cu - split-K for few output tiles, and the reduction of its partials.
//
// When a linear layer has few 256 x 256 output tiles (at most 16: up to 256
// rows at N = 4096, for 76 CTA pairs), the CTA-pair GEMM splits each tile's
// K range over several pairs and
// writes fp32 partials; this kernel adds them in split order (so the result is
// the same on every call), adds the bias, rounds once to bf16 and writes the
// output and/or its MXFP8 hand-off, exactly as the GEMM epilogue would.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

namespace mx {

namespace {

// One thread per 8 consecutive outputs of a row (N % 8 == 0): the two float4
// of every split are loaded first (splits <= kMaxSplits), then added in the
// order s = 0 .. S-1, so a call's latency is about one round trip to L2.  With
// the hand-off (N % 32 == 0), the four threads of a 32-element block are four
// consecutive lanes and quantise it together (quantize_quarter_block: the
// same bytes as quantize_block32); every lane of a warp takes part.
constexpr int kMaxSplits = 8;

template <bool kHandOff>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int S, int64_t plane,
                                                            int64_t nq, int NQ, int M, int N,
                                                            const __nv_bfloat16* __restrict__ bias,
                                                            __nv_bfloat16* __restrict__ out, uint8_t* __restrict__ yq,
                                                            uint8_t* __restrict__ ysf, int RTY, int KTY) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = t < nq;
  const int64_t row = valid ? t / NQ : 0;  // b * M + m
  const int n0 = static_cast<int>(valid ? t - row * NQ : 0) * 8;
  const int64_t base = row * N + n0;
  // launched with programmatic serialization after the GEMM that writes the
  // partials: the bias (a weight-side input) is read before the wait, the
  // partials after it
  uint4 braw = make_uint4(0, 0, 0, 0);
  if (valid && bias != nullptr) braw = __ldg(reinterpret_cast<const uint4*>(bias + n0));
  grid_dependency_wait();
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (valid) {
    float4 v[2 * kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      if (s < S) {
        const float4* ps = reinterpret_cast<const float4*>(part + s * plane + base);
        v[2 * s] = __ldg(ps);
        v[2 * s + 1] = __ldg(ps + 1);
      }
    }
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
      if (s < S) {
        acc[0] += v[2 * s].x;
        acc[1] += v[2 * s].y;
        acc[2] += v[2 * s].z;
        acc[3] += v[2 * s].w;
        acc[4] += v[2 * s + 1].x;
        acc[5] += v[2 * s + 1].y;
        acc[6] += v[2 * s + 1].z;
        acc[7] += v[2 * s + 1].w;
      }
    }
    if (bias != nullptr) {
      const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(bw[i] << 16);
        acc[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
      }
    }
  }
  const uint4 o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                             pack_bf16x2(acc[6], acc[7]));
  if (valid && out != nullptr) *reinterpret_cast<uint4*>(out + base) = o;
  if (kHandOff) {
    uint2 codes;
    const uint32_t sbyte = quantize_quarter_block(o, codes);
    if (valid) {
      *reinterpret_cast<uint2*>(yq + base) = codes;
      if ((n0 & 31) == 0) {
        const int64_t b = row / M;
        const int m = static_cast<int>(row - b * M);
        ysf[sf_packed_offset(b, m, n0 / 32, RTY, KTY)] = static_cast<uint8_t>(sbyte);
      }
    }
  }
}

}  // namespace

int splitk_splits(int64_t B, int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = B * ceil_div(M, 256) * ceil_div(N, 256);
  const int64_t kt = K / 128;
  // measured at N = K = 4096 (one call, L2 flushed / in a CUDA graph):
  // 16 tiles split 4 ways 29.4 -> 23.6 / 20.1 -> 16.0 us at M = 128, but
  // 32 tiles split 2 ways 29.3 -> 31.7 / 21.0 -> 22.2 us at M = 512; with a
  // long K (>= 64 K tiles) 32 tiles gain from 2 ways: N = 4096, K = 14336
  // (graph) 50.8 -> 39.8 us at M = 512, 49.4 -> 37.0 at M = 300; K = 8192,
  // M = 512: 32.4 -> 29.5 us
  if (tiles <= 0 || tiles > (kt >= 64 ? 32 : 16)) return 1;
  int64_t s = 64 / tiles;
  if (s > kt / 4) s = kt / 4;
  if (s > 8) s = 8;
  return s >= 2 ? static_cast<int>(s) : 1;
}

cudaError_t launch_splitk_reduce(const float* part, int splits, int64_t B, int64_t M, int64_t N, const void* bias,
                                 void* out, uint8_t* yq, uint8_t* ysf, int sms, cudaStream_t stream) {
  (void)sms;
  if (splits > kMaxSplits) return cudaErrorInvalidValue;  // splitk_splits never returns more
  const int64_t NQ = N / 8;
  const int64_t nq = B * M * NQ;
  if (nq == 0) return cudaSuccess;
  const int64_t grid = (nq + 255) / 256;
  const int RTY = static_cast<int>(ceil_div(M, kAtomRows)), KTY = static_cast<int>(ceil_div(N, kTileK));
  auto kern = yq != nullptr ? splitk_reduce_kernel<true> : splitk_reduce_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, part, splits, B * M * N, nq, static_cast<int>(NQ), static_cast<int>(M),
                            static_cast<int>(N), static_cast<const __nv_bfloat16*>(bias),
                            static_cast<__nv_bfloat16*>(out), yq, ysf, RTY, KTY);
}

}  // namespace mx
