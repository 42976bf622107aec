// gemm.cu - block-scaled MXFP8 GEMM on the 5th-generation tensor cores.
//
// out[b, m, n] = bf16( sum_k (xq[b,m,k] * 2^(sx[b,m,k/32]-127)) *
//                             (wq[b,n,k] * 2^(sw[b,n,k/32]-127)) + bias[n] )
// i.e. the block-scaled product of "AiterFlyDSLMxfp8LinearKernel.apply_weights"
// (aiter_flydsl page) followed by its bias add, with "Mxfp8LinearLayerConfig.
// bmm_batch_size" as an extra grid dimension.
//
// One persistent CTA per SM walks 128 x BN output tiles.  Warp roles:
//   warp 0      TMA producer: A / W tiles (128-byte swizzle) and scale atoms
//               into a STAGES-deep shared-memory ring;
//   warp 1      allocates tensor memory; one lane issues tcgen05.cp (scales to
//               TMEM) and tcgen05.mma kind::mxf8f6f4 block_scale (K = 32 per
//               instruction, 4 per 128-wide K tile, scale byte selected by the
//               instruction descriptor's scale-factor id);
//   warps 2..9  epilogue: two warps per 32-lane TMEM quarter, each copies its
//               half of the fp32 accumulator row (BN/2 columns) into registers,
//               hands the accumulator back to the MMA warp at once, then adds
//               the bias, rounds to bf16 and stores while the next tile's
//               main loop already runs.
// Every wait is bounded (mx_ptx.cuh); on expiry the roles stop, the kernel
// drains its own in-flight copies and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"

namespace mx {

namespace {

constexpr int BM = 128;
constexpr int BK = 128;  // bytes = E4M3 elements per K tile; one swizzle row

template <int BN_, int STAGES_>
struct Cfg {
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int NB_ATOMS = BN / kAtomRows;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFA_BYTES = kAtomBytes;
  static constexpr int SFB_BYTES = NB_ATOMS * kAtomBytes;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 2;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  // tensor memory columns: accumulator, then per-stage scale slots
  static constexpr int T_ACC = 0;
  static constexpr int T_SFA = BN;
  static constexpr int T_SFB = T_SFA + STAGES * 4;
  static constexpr int T_END = T_SFB + STAGES * NB_ATOMS * 4;
  static constexpr int TMEM_COLS = T_END <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // accumulator columns per epilogue thread
  static constexpr int THREADS = 64 + EPI_THREADS;
  static_assert(T_END <= 512, "tensor memory overflow");
  static_assert(SMEM_ALLOC <= 232448, "shared memory overflow");
  static_assert(BN % 128 == 0 && BN <= 256, "BN");
};

struct Args {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  int B, M, N, K;
  int MT, NT, KT;  // output tiles along M and N, K tiles
  int RTA, RTB;    // 128-row atom tiles of A and of W
  int total_tiles;
};

__device__ __forceinline__ void tile_coords(int tile, const Args& a, int& b, int& mt, int& nt) {
  const int per_b = a.MT * a.NT;
  b = tile / per_b;
  const int t = tile - b * per_b;
  nt = t / a.MT;
  mt = t - nt * a.MT;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gemm_mxf8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::EPI_THREADS);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < args.total_tiles; tile += gridDim.x) {
        int b, mt, nt;
        tile_coords(tile, args, b, mt, nt);
        const int nb_atoms = min(C::NB_ATOMS, args.RTB - nt * C::NB_ATOMS);
        const uint32_t tx = C::A_BYTES + C::B_BYTES + C::SFA_BYTES + nb_atoms * kAtomBytes;
        for (int kt = 0; kt < args.KT; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_3d(smem + C::OFF_A + stage * C::A_BYTES, &tmA, &full[stage], kt * BK, mt * BM, b);
          tma_load_3d(smem + C::OFF_B + stage * C::B_BYTES, &tmB, &full[stage], kt * BK,
                      nt * C::BN, b);
          const int64_t arow = static_cast<int64_t>(b) * args.KT + kt;
          bulk_load(smem + C::OFF_SFA + stage * C::SFA_BYTES,
                    args.sfa + (arow * args.RTA + mt) * kAtomBytes, C::SFA_BYTES, &full[stage]);
          bulk_load(smem + C::OFF_SFB + stage * C::SFB_BYTES,
                    args.sfb + (arow * args.RTB + static_cast<int64_t>(nt) * C::NB_ATOMS) * kAtomBytes,
                    nb_atoms * kAtomBytes, &full[stage]);
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA can exit.
        for (int s = 0; s < C::STAGES; ++s) {
          if (issued <= s) continue;
          const int64_t last = ((issued - 1 - s) / C::STAGES) * C::STAGES + s;
          mbar_wait(&full[s], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t idesc0 = idesc_mxf8(BM, C::BN);
      for (int tile = blockIdx.x; ok && tile < args.total_tiles; tile += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < args.KT; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + C::OFF_A + stage * C::A_BYTES);
          const uint32_t sb = smem_u32(smem + C::OFF_B + stage * C::B_BYTES);
          const uint32_t ssfa = smem_u32(smem + C::OFF_SFA + stage * C::SFA_BYTES);
          const uint32_t ssfb = smem_u32(smem + C::OFF_SFB + stage * C::SFB_BYTES);
          const uint32_t t_sfa = tmem + C::T_SFA + stage * 4;
          const uint32_t t_sfb = tmem + C::T_SFB + stage * C::NB_ATOMS * 4;
          tc_cp_sf(t_sfa, sdesc_sf(ssfa));
#pragma unroll
          for (int j = 0; j < C::NB_ATOMS; ++j) tc_cp_sf(t_sfb + 4 * j, sdesc_sf(ssfb + j * kAtomBytes));
          const uint64_t ad = sdesc_kmajor_sw128(sa);
          const uint64_t bd = sdesc_kmajor_sw128(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // advance 32 bytes along K inside the 128-byte swizzle row
            tc_mma_mxf8(tmem + C::T_ACC, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc0, kk, kk),
                        t_sfa, t_sfb, (kt | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) __nanosleep(200000);  // let issued tensor-core work retire
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                 // TMEM lane quarter this warp may access
    const int col0 = ((warp - 2) >> 2) * C::EPI_COLS;
    const int row = quad * 32 + lane;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < args.total_tiles; tile += gridDim.x) {
      int b, mt, nt;
      tile_coords(tile, args, b, mt, nt);
      if (!mbar_wait(acc_full, acc_phase, abort_flag)) break;
      tc_fence_after();
      uint32_t r[C::EPI_COLS];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::T_ACC + col0;
#pragma unroll
      for (int c = 0; c < C::EPI_COLS / 32; ++c)
        tmem_ld_32x32b_x32(taddr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(acc_empty);                  // accumulator free for the next tile
      acc_phase ^= 1u;

      const int m = mt * BM + row;
      if (m < args.M) {
        __nv_bfloat16* orow = args.out + (static_cast<int64_t>(b) * args.M + m) * args.N;
#pragma unroll
        for (int g = 0; g < C::EPI_COLS / 8; ++g) {
          const int n = nt * C::BN + col0 + 8 * g;
          if (n < args.N) {
            float bv[8];
            if (args.bias != nullptr) {
              const uint4 braw = *reinterpret_cast<const uint4*>(args.bias + n);
              const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                bv[2 * i] = __uint_as_float(bw[i] << 16);
                bv[2 * i + 1] = __uint_as_float(bw[i] & 0xFFFF0000u);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) bv[i] = 0.f;
            }
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(r[8 * g + 0]) + bv[0], __uint_as_float(r[8 * g + 1]) + bv[1]);
            o.y = pack_bf16x2(__uint_as_float(r[8 * g + 2]) + bv[2], __uint_as_float(r[8 * g + 3]) + bv[3]);
            o.z = pack_bf16x2(__uint_as_float(r[8 * g + 4]) + bv[4], __uint_as_float(r[8 * g + 5]) + bv[5]);
            o.w = pack_bf16x2(__uint_as_float(r[8 * g + 6]) + bv[6], __uint_as_float(r[8 * g + 7]) + bv[7]);
            *reinterpret_cast<uint4*>(orow + n) = o;
          }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

using PrefillCfg = Cfg<256, 4>;

cudaError_t make_map(CUtensorMap* map, const uint8_t* base, int64_t B, int64_t rows, int64_t K,
                     int box_rows, const char** msg) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows * K)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected an operand";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_prefill(const GemmProblem& p, int sms, cudaStream_t stream, const char** msg) {
  using C = PrefillCfg;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_mxf8_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) {
      *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return e;
    }
    attr_set[dev] = true;
  }
  CUtensorMap ma, mb;
  cudaError_t e = make_map(&ma, p.a, p.B, p.M, p.K, BM, msg);
  if (e != cudaSuccess) return e;
  e = make_map(&mb, p.w, p.B, p.N, p.K, C::BN, msg);
  if (e != cudaSuccess) return e;

  Args a;
  a.sfa = p.sfa;
  a.sfb = p.sfb;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.B = static_cast<int>(p.B);
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.MT = static_cast<int>(ceil_div(p.M, BM));
  a.NT = static_cast<int>(ceil_div(p.N, C::BN));
  a.KT = static_cast<int>(p.K / BK);
  a.RTA = static_cast<int>(ceil_div(p.M, kAtomRows));
  a.RTB = static_cast<int>(ceil_div(p.N, kAtomRows));
  a.total_tiles = a.B * a.MT * a.NT;
  const int grid = a.total_tiles < sms ? a.total_tiles : sms;
  gemm_mxf8_kernel<C><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(ma, mb, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) *msg = "GEMM launch failed";
  return e;
}

cudaError_t take_status_gemm(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
