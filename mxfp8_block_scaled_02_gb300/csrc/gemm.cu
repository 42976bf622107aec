// gemm.cu - block-scaled MXFP8 GEMM on the 5th-generation tensor cores.
//
// out[b, m, n] = bf16( sum_k (xq[b,m,k] * 2^(sx[b,m,k/32]-127)) *
//                             (wq[b,n,k] * 2^(sw[b,n,k/32]-127)) + bias[n] )
// i.e. the block-scaled product of "AiterFlyDSLMxfp8LinearKernel.apply_weights"
// (aiter_flydsl page) followed by its bias add, with "Mxfp8LinearLayerConfig.
// bmm_batch_size" as an extra grid dimension.
//
// Serves M <= 128 when the fused small-M path does not apply (path 2 forces
// it); M > 128 goes to the CTA-pair kernel of gemm_pair.cu.
// One persistent CTA per SM walks 128 x BN output tiles.  Warp roles:
//   warp 0       TMA producer: A / W tiles (128-byte swizzle) and scale atoms
//                into a STAGES-deep shared-memory ring; the atoms complete on
//                their own barrier so their trip to TMEM overlaps the
//                operand load;
//   warp 1       allocates tensor memory; one lane issues tcgen05.mma
//                kind::mxf8f6f4 block_scale (K = 32 per instruction, 4 per
//                128-wide K tile, the scale byte picked by the instruction
//                descriptor's scale-factor id);
//   warps 2..5   scale-factor writers, one per 32-lane TMEM quarter: each lane
//                moves one 16-byte line of the stage's scale atoms from shared
//                memory into its TMEM lane with tcgen05.st (every quarter gets
//                the same lines).  Doing this with warps rather than tcgen05.cp
//                keeps the copies off the tensor pipe, which runs MMAs and
//                copies in order;
//   warps 6..13  epilogue, two warps per TMEM quarter, each BN/2 columns: copy
//                the fp32 accumulator out of TMEM 32 columns at a time, add the
//                bias and round to bf16 at once, hand the accumulator back to
//                the MMA warp, then write the bf16 rows through a 2 KB shared
//                staging buffer with TMA bulk-tensor stores (which also clip
//                the M / N edges), while the next tile's main loop runs.
// Every wait is bounded (mx_ptx.cuh); on expiry the roles stop, the kernel
// drains its own in-flight copies and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_epilogue.cuh"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

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
  static constexpr int SF_WARPS = 4;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // accumulator columns per epilogue thread
  static constexpr int STAGE_OUT = 32 * 32 * 2;          // one 32 x 32 bf16 box per epilogue warp
  static constexpr int THREADS = 64 + SF_WARPS * 32 + EPI_THREADS;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_OUT = OFF_SFB + STAGES * SFB_BYTES;
  static constexpr int OFF_BIAS = OFF_OUT + EPI_WARPS * STAGE_OUT;  // per epilogue warp: its EPI_COLS bias values
  static constexpr int OFF_BAR = OFF_BIAS + EPI_WARPS * EPI_COLS * 2;
  // per stage: full (operands), sf_full (scale atoms), sf_ready, empty; then acc_full/empty
  static constexpr int NUM_BARS = 4 * STAGES + 2;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
  // tensor memory columns: accumulator, then per-stage scale slots
  static constexpr int T_ACC = 0;
  static constexpr int T_SFA = BN;
  static constexpr int T_SFB = T_SFA + STAGES * 4;
  static constexpr int T_END = T_SFB + STAGES * NB_ATOMS * 4;
  static constexpr int TMEM_COLS = T_END <= 256 ? 256 : 512;
  // columns the epilogue's warm-up pass reads (allocated, never written)
  static constexpr int T_WARM = TMEM_COLS - EPI_COLS;
  static_assert(T_END <= 512, "tensor memory overflow");
  static_assert(T_WARM >= T_END, "the warm-up columns must be unused");
  static_assert(SMEM_ALLOC <= 232448, "shared memory overflow");
  static_assert(BN % 128 == 0 && BN <= 256, "BN");
  static_assert(EPI_COLS % 32 == 0, "epilogue chunks");
  static_assert(EPI_COLS == 128, "the MXFP8 hand-off quantises 128 columns (one scale word) per thread");
};

struct Args {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const __nv_bfloat16* bias;
  uint8_t* yq;   // MXFP8 hand-off outputs (nullptr: none), see mx_epilogue.cuh
  uint8_t* ysf;
  int B, M, N, K;
  int MT, NT, KT;  // output tiles along M and N, K tiles
  int RTA, RTB;    // 128-row atom tiles of A and of W
  int RTY, KTY;    // atom tiles of the hand-off scales (rows, K tiles = N / 128)
  int store_bf16;  // 0: the bf16 output is not written
  int wfmt;        // weight (B operand) element format
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
                     const __grid_constant__ CUtensorMap tmOut, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* sf_full = full + C::STAGES;
  uint64_t* sf_ready = sf_full + C::STAGES;
  uint64_t* empty = sf_ready + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], C::SF_WARPS);  // one arrive per writer warp
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, C::EPI_WARPS);  // one arrive per epilogue warp
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmOut);
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
        const uint32_t sf_tx = C::SFA_BYTES + nb_atoms * kAtomBytes;
        for (int kt = 0; kt < args.KT; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // The scale atoms get their own barrier: they land long before the
          // operands, so the writers put them in TMEM while the operands load.
          const int64_t arow = static_cast<int64_t>(b) * args.KT + kt;
          mbar_arrive_expect_tx(&sf_full[stage], sf_tx);
          bulk_load(smem + C::OFF_SFA + stage * C::SFA_BYTES,
                    args.sfa + (arow * args.RTA + mt) * kAtomBytes, C::SFA_BYTES, &sf_full[stage]);
          bulk_load(smem + C::OFF_SFB + stage * C::SFB_BYTES,
                    args.sfb + (arow * args.RTB + static_cast<int64_t>(nt) * C::NB_ATOMS) * kAtomBytes,
                    nb_atoms * kAtomBytes, &sf_full[stage]);
          mbar_arrive_expect_tx(&full[stage], C::A_BYTES + weight_tile_tx_bytes(C::BN, args.wfmt));
          tma_load_3d(smem + C::OFF_A + stage * C::A_BYTES, &tmA, &full[stage], kt * BK, mt * BM, b);
          tma_load_3d(smem + C::OFF_B + stage * C::B_BYTES, &tmB, &full[stage], kt * BK,
                      nt * C::BN, b);
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
          mbar_wait(&sf_full[s], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr);
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
      const uint32_t idesc0 = idesc_with_types(idesc_mxf8(BM, C::BN), kFmtE4M3, args.wfmt);
      for (int tile = blockIdx.x; ok && tile < args.total_tiles; tile += gridDim.x) {
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < args.KT; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag) || !mbar_wait(&sf_ready[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(smem + C::OFF_A + stage * C::A_BYTES));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(smem + C::OFF_B + stage * C::B_BYTES));
          const uint32_t t_sfa = tmem + C::T_SFA + stage * 4;
          const uint32_t t_sfb = tmem + C::T_SFB + stage * C::NB_ATOMS * 4;
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
  } else if (warp < 2 + C::SF_WARPS) {
    // ------------------------------------------------------------ scale-factor writers
    // Atom line `lane` holds rows {lane, lane+32, lane+64, lane+96} x 4 blocks;
    // the MMA reads it from every 32-lane quarter, so each quarter gets a copy.
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = blockIdx.x; tile < args.total_tiles; tile += gridDim.x) {
      bool ok = true;
      for (int kt = 0; kt < args.KT; ++kt) {
        if (!mbar_wait(&sf_full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint4 va = *reinterpret_cast<const uint4*>(smem + C::OFF_SFA + stage * C::SFA_BYTES + lane * 16);
        tmem_st_32x32b_x4(lane_base + C::T_SFA + stage * 4, va.x, va.y, va.z, va.w);
#pragma unroll
        for (int j = 0; j < C::NB_ATOMS; ++j) {
          const uint4 vb = *reinterpret_cast<const uint4*>(smem + C::OFF_SFB + stage * C::SFB_BYTES +
                                                           j * kAtomBytes + lane * 16);
          tmem_st_32x32b_x4(lane_base + C::T_SFB + (stage * C::NB_ATOMS + j) * 4, vb.x, vb.y, vb.z, vb.w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2 - C::SF_WARPS;     // 0 .. EPI_WARPS-1
    const int quad = warp & 3;                 // TMEM lane quarter this warp may access
    const int col0 = (ew >> 2) * C::EPI_COLS;
    uint8_t* stage_out = smem + C::OFF_OUT + ew * C::STAGE_OUT;
    uint4* bias_s = reinterpret_cast<uint4*>(smem + C::OFF_BIAS + ew * C::EPI_COLS * 2);
    uint32_t acc_phase = 0;
    bool pending = false;  // lane 0: a bulk store of this warp may still read stage_out
    // The first pass (live == false) is a warm-up: it runs the drain and
    // store code below once, on tensor-memory columns nothing writes, with
    // every wait, arrive and global write skipped, so that this code is in
    // the SM's instruction cache when the first accumulator is ready (a
    // first drain otherwise waits on instruction fetches from DRAM).  The
    // pass count starts from an opaque register so that one copy of the body
    // serves both.
    int pass;
    asm volatile("mov.s32 %0, -1;" : "=r"(pass));
    for (int tile = blockIdx.x; tile < args.total_tiles; ++pass) {
      const bool live = pass >= 0;
      int b, mt, nt;
      tile_coords(tile, args, b, mt, nt);
      if (live) tile += gridDim.x;
      if (live && args.bias != nullptr) {
        // this warp's bias values (zero past N) into shared memory while the
        // tile's MMAs run, so that the drain below reads no global memory
        if (lane < C::EPI_COLS / 8) {
          const int n = nt * C::BN + col0 + 8 * lane;
          bias_s[lane] = n < args.N ? *reinterpret_cast<const uint4*>(args.bias + n) : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      if (live) {
        if (!mbar_wait(acc_full, acc_phase, abort_flag)) break;
        tc_fence_after();
      }
      // accumulator -> registers as bf16 (bias added in fp32, one rounding)
      uint32_t packed[C::EPI_COLS / 2];
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(quad * 32) << 16) + (live ? C::T_ACC + col0 : C::T_WARM);
#pragma unroll
      for (int c = 0; c < C::EPI_COLS / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float bv[8];
          if (args.bias != nullptr) {
            const uint4 braw = bias_s[c * 4 + g];
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
#pragma unroll
          for (int i = 0; i < 4; ++i)
            packed[c * 16 + g * 4 + i] = pack_bf16x2(__uint_as_float(r[8 * g + 2 * i]) + bv[2 * i],
                                                     __uint_as_float(r[8 * g + 2 * i + 1]) + bv[2 * i + 1]);
        }
      }
      if (live) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);   // accumulator free for the next tile
        acc_phase ^= 1u;
      }

      // the same bf16 values quantised for the next layer (MXFP8 hand-off)
      if (live && args.yq != nullptr)
        store_quantized_row128(packed, args.yq, args.ysf, b, mt * BM + quad * 32 + lane, nt * C::BN + col0,
                               args.M, args.N, args.RTY, args.KTY);
      if (!args.store_bf16) continue;
      // registers -> 32 x 32 staging box -> TMA store (rows/columns past M, N are clipped)
#pragma unroll
      for (int c = 0; c < C::EPI_COLS / 32; ++c) {
        if (lane == 0 && pending) bulk_wait_group_read0();
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(stage_out + lane * 64);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(packed[c * 16 + 4 * q], packed[c * 16 + 4 * q + 1], packed[c * 16 + 4 * q + 2],
                              packed[c * 16 + 4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && live) {
          tma_store_3d(&tmOut, stage_out, nt * C::BN + col0 + c * 32, mt * BM + quad * 32, b);
          bulk_commit_group();
          pending = true;
        }
      }
    }
    if (lane == 0 && pending) bulk_wait_group0();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

using PrefillCfg = Cfg<256, 4>;

}  // namespace

// bf16 [B][M][N] output, box {32 columns, 32 rows, 1}, no swizzle.
cudaError_t make_output_map(CUtensorMap* map, void* out, int64_t B, int64_t M, int64_t N, const char** msg) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N * 2), static_cast<cuuint64_t>(M * N * 2)};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected the output";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t make_partial_map(CUtensorMap* map, float* part, int64_t Z, int64_t M, int64_t N, const char** msg) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(Z)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N * 4), static_cast<cuuint64_t>(M * N * 4)};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected the split-K partials";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// 3-D map over [B][rows][K] bytes, box {128, box_rows, 1}, 128-byte swizzle,
// zero fill outside the tensor.
cudaError_t make_operand_map(CUtensorMap* map, const uint8_t* base, int64_t B, int64_t rows,
                             int64_t K, int box_rows, const char** msg, int fmt) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  // element counts along K; the row stride is in bytes (3K/4 for packed FP6)
  const int64_t row_bytes = fmt == 0 ? K : K * 3 / 4;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows * row_bytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dtype = fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
  CUresult r = encode(map, dtype, 3, const_cast<uint8_t*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected an operand";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

bool gemm_prefill_uses_pair(const GemmProblem& p, int sms) {
  // 256 x 256 tiles on CTA pairs load 32 KB per SM and K tile against 48 KB
  // for 128 x 256 tiles on one CTA, and measure faster once M spans a pair tile.
  // Up to 128 rows the layer is bound by streaming the weights: there pairs
  // are used while one wave of them holds every tile, which puts twice as
  // many SMs on the stream (3-15 % faster at M = 16..128, N = 4096..14336).
  const bool one_wave_of_pairs = p.B * ceil_div(p.N, 256) * 2 <= sms;
  return p.tiles == 2 ||
         (p.tiles == 0 && (p.M > 128 || one_wave_of_pairs || (p.part != nullptr && p.splits > 1)) && sms >= 2);
}

cudaError_t launch_gemm_prefill(const GemmProblem& p, int sms, cudaStream_t stream, const char** msg) {
  if (gemm_prefill_uses_pair(p, sms)) return launch_gemm_pair(p, sms, stream, msg);
  if (p.sfa_rowmajor) {
    *msg = "row-major activation scales need the CTA-pair kernel";
    return cudaErrorInvalidValue;
  }
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
  CUtensorMap ma, mb, mo;
  cudaError_t e = make_operand_map(&ma, p.a, p.B, p.M, p.K, BM, msg);
  if (e != cudaSuccess) return e;
  e = make_operand_map(&mb, p.w, p.B, p.N, p.K, C::BN, msg, p.wfmt);
  if (e != cudaSuccess) return e;
  // without a bf16 output the map is never used; any aligned address will do
  e = make_output_map(&mo, p.out != nullptr ? p.out : static_cast<void*>(p.yq), p.B, p.M, p.N, msg);
  if (e != cudaSuccess) return e;

  Args a;
  a.sfa = p.sfa;
  a.sfb = p.sfb;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.yq = p.yq;
  a.ysf = p.ysf;
  a.RTY = static_cast<int>(ceil_div(p.M, kAtomRows));
  a.KTY = static_cast<int>(ceil_div(p.N, kTileK));
  a.store_bf16 = p.out != nullptr;
  a.wfmt = p.wfmt;
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
  gemm_mxf8_kernel<C><<<grid, C::THREADS, C::SMEM_ALLOC, stream>>>(ma, mb, mo, a);
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
