// quantize.cu - dynamic MXFP8 quantisation and the scale-factor repack.
//
// The per-block arithmetic (OCP MX v1.0, section 6.3) lives in mx_quant.cuh,
// shared with the fused small-M GEMM so that both produce the same bytes.
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
constexpr int kQuantUnroll = 4;  // 8-block tasks per work item, loads all in flight

// A task is 8 consecutive 32-element blocks of one row (256 values, 512
// bytes of bf16); lane l owns 8 values: block j = l / 4 of the task, quarter
// l % 4 of that block, and four lanes combine their amax by shuffles.  A work
// item is kQuantUnroll consecutive tasks of one row, so the row (and, for the
// packed layout, its batch and atom row) is found with one division per item.
// kPacked selects the scale output: false = row-major [rows, K/32], true = the
// 512-byte atom layout of mx_layout.cuh (rows grouped per batch of rows_per_b).
template <bool kPacked>
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(
    const uint4* __restrict__ x, uint32_t KB, uint32_t tasks_per_row, uint32_t items_per_row,
    uint32_t nitems, uint8_t* __restrict__ q, uint8_t* __restrict__ s, uint32_t rows_per_b,
    uint32_t RT, uint32_t KT) {
  // The GEMM that follows may start its prologue and weight loads now; it
  // waits for this grid to finish before it reads the codes and scales.
  launch_dependents();
  const int lane = threadIdx.x & 31;
  const uint32_t j = lane >> 2, part = lane & 3;
  const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const int64_t atom_k_stride = static_cast<int64_t>(RT) * kAtomBytes;  // next K tile, same rows

  for (uint32_t item = warp; item < nitems; item += nwarps) {
    const uint32_t row = item / items_per_row;
    const uint32_t t0 = (item - row * items_per_row) * kQuantUnroll;
    const int64_t row_blk = static_cast<int64_t>(row) * KB;  // first block of the row
    uint4 v[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const uint32_t kb = (t0 + u) * 8 + j;
      const bool valid = t0 + u < tasks_per_row && kb < KB;
      v[u] = valid ? __ldg(x + (row_blk + kb) * 4 + part) : make_uint4(0, 0, 0, 0);
    }
    int64_t atom_row = 0;  // packed: offset of (row, block 0) in its first atom
    if (kPacked) {
      const uint32_t b = row / rows_per_b, r = row - b * rows_per_b;
      atom_row = (static_cast<int64_t>(b) * KT * RT + (r >> 7)) * kAtomBytes + (r & 31) * 16 +
                 ((r >> 5) & 3) * 4;
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const uint32_t task = t0 + u;
      const uint32_t kb_task = task * 8;
      const uint32_t kb = kb_task + j;
      const bool valid = task < tasks_per_row && kb < KB;
      uint2 codes;
      const uint32_t sbyte = quantize_quarter_block(v[u], codes);
      if (valid) *reinterpret_cast<uint2*>(q + (row_blk + kb) * 32 + part * 8) = codes;

      // Scale bytes: gather the task's 8 bytes (lanes 0, 4, ..., 28) so that
      // whole words are stored when the task is complete.
      const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, sbyte, (lane & 16) + 0);
      const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, sbyte, (lane & 16) + 4);
      const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, sbyte, (lane & 16) + 8);
      const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, sbyte, (lane & 16) + 12);
      const uint32_t word = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
      const bool full_task = task < tasks_per_row && kb_task + 8 <= KB;
      if (kPacked) {
        // blocks kb..kb+3 (kb % 4 == 0) are 4 consecutive bytes of one atom
        if (full_task) {
          if ((lane & 15) == 0)
            *reinterpret_cast<uint32_t*>(s + atom_row + (kb >> 2) * atom_k_stride) = word;
        } else if (valid && part == 0) {
          s[atom_row + (kb >> 2) * atom_k_stride + (kb & 3)] = static_cast<uint8_t>(sbyte);
        }
      } else {
        const uint32_t hi_word = __shfl_sync(0xFFFFFFFFu, word, 16);
        const int64_t off = row_blk + kb_task;
        if (full_task && (off & 7) == 0) {
          if (lane == 0) *reinterpret_cast<uint2*>(s + off) = make_uint2(word, hi_word);
        } else if (valid && part == 0) {
          s[row_blk + kb] = static_cast<uint8_t>(sbyte);
        }
      }
    }
  }
}

// Row-major [B, R, KB] -> packed atoms; one thread per 4 output bytes (the 4
// blocks of one row inside an atom).  Padding rows/blocks are written as 0.
__global__ void __launch_bounds__(256) sf_pack_kernel(const uint8_t* __restrict__ src, int64_t R,
                                                       int64_t KB, int64_t RT, int64_t KT,
                                                       uint32_t* __restrict__ dst, int64_t nwords) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t wi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; wi < nwords;
       wi += stride) {
    const int64_t atom = wi >> 7;          // 128 words per 512-byte atom
    const int within = static_cast<int>(wi & 127);
    const int line = within >> 2, grp = within & 3;
    const int64_t rt = atom % RT;
    const int64_t kt = (atom / RT) % KT;
    const int64_t b = atom / (RT * KT);
    const int64_t r = rt * kAtomRows + grp * 32 + line;
    uint32_t v = 0;
    if (r < R) {
      const uint8_t* row = src + (b * R + r) * KB;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t kb = kt * 4 + j;
        if (kb < KB) v |= static_cast<uint32_t>(row[kb]) << (8 * j);
      }
    }
    dst[wi] = v;
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

cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                            bool packed_scales, int64_t B, int64_t rows_per_b, int sms,
                            cudaStream_t stream) {
  (void)B;
  const int64_t KB = K / 32;
  const int64_t tasks_per_row = ceil_div(KB, 8);
  const int64_t items_per_row = ceil_div(tasks_per_row, kQuantUnroll);
  const int64_t nitems = rows * items_per_row;
  if (nitems == 0) return cudaSuccess;
  if (nitems > 0x7FFFFFFFll || KB > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  static int per_sm[2] = {0, 0};
  int& occ = per_sm[packed_scales ? 1 : 0];
  if (occ == 0) {
    cudaError_t e = packed_scales
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quantize_kernel<true>, kQuantThreads, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, quantize_kernel<false>, kQuantThreads, 0);
    if (e != cudaSuccess || occ < 1) occ = 1;
  }
  const int grid = grid_for(nitems * 32, kQuantThreads, sms, occ);
  const uint32_t RT = static_cast<uint32_t>(ceil_div(rows_per_b, kAtomRows));
  const uint32_t KT = static_cast<uint32_t>(ceil_div(K, kTileK));
  if (packed_scales)
    quantize_kernel<true><<<grid, kQuantThreads, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint32_t>(KB), static_cast<uint32_t>(tasks_per_row),
        static_cast<uint32_t>(items_per_row), static_cast<uint32_t>(nitems), q, s,
        static_cast<uint32_t>(rows_per_b), RT, KT);
  else
    quantize_kernel<false><<<grid, kQuantThreads, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint32_t>(KB), static_cast<uint32_t>(tasks_per_row),
        static_cast<uint32_t>(items_per_row), static_cast<uint32_t>(nitems), q, s,
        static_cast<uint32_t>(rows_per_b), RT, KT);
  return cudaGetLastError();
}

cudaError_t launch_sf_pack(const uint8_t* src, int64_t B, int64_t R, int64_t K, uint8_t* dst,
                           int sms, cudaStream_t stream) {
  const int64_t KB = K / 32, RT = ceil_div(R, kAtomRows), KT = ceil_div(K, kTileK);
  const int64_t nwords = sf_packed_bytes(B, R, K) / 4;
  if (nwords == 0) return cudaSuccess;
  sf_pack_kernel<<<grid_for(nwords, 256, sms, 8), 256, 0, stream>>>(
      src, R, KB, RT, KT, reinterpret_cast<uint32_t*>(dst), nwords);
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
