// quantize.cu - dynamic MXFP8 quantisation and the scale-factor repack.
//
// The per-block arithmetic (OCP MX v1.0, section 6.3) lives in mx_quant.cuh:
// this kernel uses quantize_block32 (one lane per block), the fused small-M
// GEMM quantize_quarter_block (four lanes per block); both take the same
// decisions on the same bf16 bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

namespace mx {

namespace {

constexpr int kQuantThreads = 256;
constexpr int kQU = 2;  // 32-block warp tasks per loop iteration, loads all in flight

// Block g of the flat [rows, K] array is row g / KB, block g % KB; its codes
// are bytes [32 g, 32 g + 32) of q and, in the row-major scale layout, its
// scale is byte g of s.  Lane l of a warp task takes block 32 t + l, so a warp
// reads 2 KB and writes 1 KB of codes and 32 scale bytes, contiguous.
// kPacked selects the 512-byte atom layout of mx_layout.cuh for the scales
// (rows grouped per batch of rows_per_b).  kEarly lets the next kernel in the
// stream start at once (griddepcontrol.launch_dependents): only for the
// quantise step inside the linear layer, whose GEMM reads the codes and scales
// after its own dependency wait and loads nothing this kernel writes before it.
// Those launches are programmatic too: the kernel waits for the one before it
// (griddepcontrol.wait) before its first read of x or write of anything, so
// it may be resident early behind a kernel that triggers its dependents.
// FMT selects the element format (mx_quant.cuh): E4M3, or an FP6 format for
// MXFP6 weights (row-major scales only).
template <bool kPacked, bool kEarly, int FMT = kFmtE4M3>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(
    const uint4* __restrict__ x, uint32_t total_blocks, uint32_t KB, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s, uint32_t rows_per_b, uint32_t RT, uint32_t KT) {
  if (kEarly) {
    launch_dependents();
    grid_dependency_wait();
  }
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t ntasks = (total_blocks + 31) / 32;
  const int64_t atom_k_stride = static_cast<int64_t>(RT) * kAtomBytes;  // next K tile, same rows

  for (uint32_t t0 = warp * kQU; t0 < ntasks; t0 += nwarps * kQU) {
    uint4 v[kQU][4];
#pragma unroll
    for (int u = 0; u < kQU; ++u) {
      const uint32_t g = (t0 + u) * 32 + lane;
      const bool valid = t0 + u < ntasks && g < total_blocks;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[u][k] = valid ? __ldg(x + static_cast<uint64_t>(g) * 4 + k) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQU; ++u) {
      const uint32_t g0 = (t0 + u) * 32;
      const uint32_t g = g0 + lane;
      uint4 c0, c1;
      const uint32_t sbyte = quantize_block32<FMT>(v[u], c0, c1);
      if (t0 + u >= ntasks || g >= total_blocks) continue;
      uint4* qd = reinterpret_cast<uint4*>(q + static_cast<uint64_t>(g) * 32);
      qd[0] = c0;
      qd[1] = c1;
      if (!kPacked) {
        s[g] = static_cast<uint8_t>(sbyte);
      } else {
        // row and block of the warp's first block (one division), then this lane's
        uint32_t row = g0 / KB;
        uint32_t kb = g0 - row * KB + lane;
        while (kb >= KB) {
          kb -= KB;
          ++row;
        }
        const uint32_t b = row / rows_per_b, r = row - b * rows_per_b;
        s[(static_cast<int64_t>(b) * KT * RT + (r >> 7)) * kAtomBytes + (r & 31) * 16 + ((r >> 5) & 3) * 4 +
          (kb >> 2) * atom_k_stride + (kb & 3)] = static_cast<uint8_t>(sbyte);
      }
    }
  }
}

// Row-major [B, R, KB] -> packed atoms; one thread per 4 output bytes (the 4
// blocks of one row inside an atom).  Padding rows/blocks are written as 0.
// 32-bit index arithmetic (the host checks the sizes): 64-bit divisions per
// word made this repack cost ~20 us for 3.7 MB of scales.  kEarly as for the
// quantise kernel: only the activation-scale repack inside the linear layer
// triggers its dependents early; a weight repack never does, because the GEMMs
// load weight scales before their dependency wait.
template <bool kEarly>
__global__ void __launch_bounds__(256) sf_pack_kernel(const uint8_t* __restrict__ src, uint32_t R,
                                                       uint32_t KB, uint32_t RT, uint32_t KT,
                                                       uint32_t* __restrict__ dst, uint32_t nwords) {
  if (kEarly) launch_dependents();
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t wi = blockIdx.x * blockDim.x + threadIdx.x; wi < nwords; wi += stride) {
    const uint32_t atom = wi >> 7;  // 128 words per 512-byte atom
    const uint32_t within = wi & 127;
    const uint32_t line = within >> 2, grp = within & 3;
    const uint32_t bk = atom / RT;  // b * KT + kt
    const uint32_t rt = atom - bk * RT;
    const uint32_t b = bk / KT;
    const uint32_t kt = bk - b * KT;
    const uint32_t r = rt * kAtomRows + grp * 32 + line;
    uint32_t v = 0;
    if (r < R) {
      const uint8_t* row = src + (static_cast<uint64_t>(b) * R + r) * KB;
      if ((KB & 3) == 0) {
        // the word's 4 blocks are 4 aligned bytes of the row (KB % 4 == 0 keeps
        // every row 4-byte aligned): one load instead of four
        v = __ldg(reinterpret_cast<const uint32_t*>(row + kt * 4));
      } else {
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j) {
          const uint32_t kb = kt * 4 + j;
          if (kb < KB) v |= static_cast<uint32_t>(row[kb]) << (8 * j);
        }
      }
    }
    dst[wi] = v;
  }
}

// FP6 codes, one per byte (low 6 bits) -> the packed 6-bit layout the weight
// tensor map reads (CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B): every 16
// consecutive codes of a row become 12 bytes, code i in bits [6i, 6i + 6) of
// that little-endian 96-bit group, with no gaps; a row of K codes is 3K/4
// bytes.  One thread per group of 16.
__global__ void __launch_bounds__(256) fp6_pack_kernel(const uint4* __restrict__ codes, uint32_t* __restrict__ out,
                                                       uint32_t ngroups) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < ngroups; g += stride) {
    const uint4 v = __ldg(codes + g);
    const uint32_t w[4] = {v.x & 0x3F3F3F3Fu, v.y & 0x3F3F3F3Fu, v.z & 0x3F3F3F3Fu, v.w & 0x3F3F3F3Fu};
    uint32_t c[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) c[i] = (w[i >> 2] >> (8 * (i & 3))) & 0x3Fu;
    const uint32_t o0 = c[0] | (c[1] << 6) | (c[2] << 12) | (c[3] << 18) | (c[4] << 24) | (c[5] << 30);
    const uint32_t o1 = (c[5] >> 2) | (c[6] << 4) | (c[7] << 10) | (c[8] << 16) | (c[9] << 22) | (c[10] << 28);
    const uint32_t o2 = (c[10] >> 4) | (c[11] << 2) | (c[12] << 8) | (c[13] << 14) | (c[14] << 20) | (c[15] << 26);
    out[3 * static_cast<uint64_t>(g)] = o0;
    out[3 * static_cast<uint64_t>(g) + 1] = o1;
    out[3 * static_cast<uint64_t>(g) + 2] = o2;
  }
}

// Packed atoms -> row-major [B, R, KB]; one thread per output byte.
__global__ void __launch_bounds__(256) sf_unpack_kernel(const uint8_t* __restrict__ src, int64_t B,
                                                         int64_t R, int64_t KB, int64_t RT,
                                                         int64_t KT, uint8_t* __restrict__ dst) {
  const int64_t n = B * R * KB;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t kb = i % KB;
    const int64_t r = (i / KB) % R;
    const int64_t b = i / (KB * R);
    dst[i] = src[sf_packed_offset(b, r, kb, RT, KT)];
  }
}

int grid_for(int64_t work_items, int threads, int sms, int per_sm) {
  int64_t g = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

template <bool kPacked, bool kEarly, int FMT = kFmtE4M3>
cudaError_t launch_quantize_t(const void* x, int64_t total_blocks, int64_t K, uint8_t* q, uint8_t* s,
                              int64_t rows_per_b, int sms, cudaStream_t stream) {
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kernel<kPacked, kEarly, FMT>,
                                                                  kQuantThreads, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  }
  const int64_t ntasks = ceil_div(total_blocks, 32);
  const int grid = grid_for(ceil_div(ntasks, kQU) * 32, kQuantThreads, sms, per_sm);
  const uint32_t RT = static_cast<uint32_t>(ceil_div(rows_per_b, kAtomRows));
  const uint32_t KT = static_cast<uint32_t>(ceil_div(K, kTileK));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kQuantThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kEarly ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, quantize_kernel<kPacked, kEarly, FMT>, static_cast<const uint4*>(x),
                            static_cast<uint32_t>(total_blocks), static_cast<uint32_t>(K / 32), q, s,
                            static_cast<uint32_t>(rows_per_b), RT, KT);
}

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                            bool packed_scales, int64_t B, int64_t rows_per_b, int sms,
                            cudaStream_t stream, bool early_trigger) {
  (void)B;
  const int64_t total_blocks = rows * (K / 32);
  if (total_blocks == 0) return cudaSuccess;
  if (total_blocks > kMaxBlocks32) return cudaErrorInvalidValue;  // the host refuses these first
  if (packed_scales)
    return early_trigger ? launch_quantize_t<true, true>(x, total_blocks, K, q, s, rows_per_b, sms, stream)
                         : launch_quantize_t<true, false>(x, total_blocks, K, q, s, rows_per_b, sms, stream);
  return early_trigger ? launch_quantize_t<false, true>(x, total_blocks, K, q, s, rows_per_b, sms, stream)
                       : launch_quantize_t<false, false>(x, total_blocks, K, q, s, rows_per_b, sms, stream);
}

cudaError_t launch_quantize_weights(const void* x, int64_t rows, int64_t K, int fmt, uint8_t* q, uint8_t* s,
                                    int sms, cudaStream_t stream) {
  const int64_t total_blocks = rows * (K / 32);
  if (total_blocks == 0) return cudaSuccess;
  if (total_blocks > kMaxBlocks32) return cudaErrorInvalidValue;  // the host refuses these first
  if (fmt == kFmtE2M3)
    return launch_quantize_t<false, false, kFmtE2M3>(x, total_blocks, K, q, s, rows, sms, stream);
  if (fmt == kFmtE3M2)
    return launch_quantize_t<false, false, kFmtE3M2>(x, total_blocks, K, q, s, rows, sms, stream);
  return launch_quantize_t<false, false, kFmtE4M3>(x, total_blocks, K, q, s, rows, sms, stream);
}

cudaError_t launch_fp6_pack(const uint8_t* codes, int64_t n, uint8_t* out, int sms, cudaStream_t stream) {
  const int64_t ngroups = n / 16;
  if (ngroups == 0) return cudaSuccess;
  if (ngroups > kMaxBlocks32) return cudaErrorInvalidValue;  // the host refuses these first
  fp6_pack_kernel<<<grid_for(ngroups, 256, sms, 8), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(codes), reinterpret_cast<uint32_t*>(out), static_cast<uint32_t>(ngroups));
  return cudaGetLastError();
}

cudaError_t launch_sf_pack(const uint8_t* src, int64_t B, int64_t R, int64_t K, uint8_t* dst,
                           int sms, cudaStream_t stream, bool early_trigger) {
  const int64_t KB = K / 32, RT = ceil_div(R, kAtomRows), KT = ceil_div(K, kTileK);
  const int64_t nwords = sf_packed_bytes(B, R, K) / 4;
  if (nwords == 0) return cudaSuccess;
  if (nwords > kMaxBlocks32 || B * R * KB > kMaxBlocks32) return cudaErrorInvalidValue;  // refused by the host first
  const int grid = grid_for(nwords, 256, sms, 8);
  auto kern = early_trigger ? sf_pack_kernel<true> : sf_pack_kernel<false>;
  kern<<<grid, 256, 0, stream>>>(src, static_cast<uint32_t>(R), static_cast<uint32_t>(KB),
                                 static_cast<uint32_t>(RT), static_cast<uint32_t>(KT),
                                 reinterpret_cast<uint32_t*>(dst), static_cast<uint32_t>(nwords));
  return cudaGetLastError();
}

cudaError_t launch_sf_unpack(const uint8_t* src, int64_t B, int64_t R, int64_t K, uint8_t* dst,
                             int sms, cudaStream_t stream) {
  const int64_t KB = K / 32, RT = ceil_div(R, kAtomRows), KT = ceil_div(K, kTileK);
  const int64_t n = B * R * KB;
  if (n == 0) return cudaSuccess;
  sf_unpack_kernel<<<grid_for(n, 256, sms, 8), 256, 0, stream>>>(src, B, R, KB, RT, KT, dst);
  return cudaGetLastError();
}

cudaError_t take_status_quantize(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
