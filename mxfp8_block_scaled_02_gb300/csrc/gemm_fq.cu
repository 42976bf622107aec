// gemm_fq.cu - the MXFP8 linear layer with the activation quantisation fused
// into the GEMM, for shapes whose 128 x 256 output tiles all fit on the GPU at
// once and whose activation rows few output tiles share (N <= 512): the
// batched shape of "Mxfp8LinearLayerConfig.bmm_batch_size".
//
// Same function as the quantise kernel followed by the one-CTA GEMM (the
// mxfp8_e4m3_quantize step, then the block-scaled product and the bias add of
// "AiterFlyDSLMxfp8LinearKernel.apply_weights", aiter_flydsl page), and the
// same bytes: the same per-block quantiser (quantize_block32) writes the codes
// and scales that the same MMA shape reads.  What changes is the traffic.  At
// B = 16, M = N = 512, K = 7168 the unfused layer reads x (117 MB bf16), writes
// its E4M3 copy (59 MB) and reads that copy back, next to the 59 MB of weights;
// here x is read once, into shared memory, and its codes never leave the SM.
//
// One CTA per 128 x 256 output tile (the host launches exactly that many):
//   warp 0       TMA producer: per 128-wide K tile, the tile's x rows as bf16
//                (two 64-column boxes, 128-byte swizzle) into a 2-slot staging
//                ring, and the 256 weight rows plus their two scale atoms into
//                a 3-slot operand ring; the first weight round goes out before
//                griddepcontrol.wait (weights do not depend on the previous
//                kernel in the stream), every x copy after it;
//   warp 1       TMEM allocation; one lane issues the MMAs;
//   warps 2..17  quantiser: thread t takes row t % 128 and block t / 128 of
//                the K tile, reads its 64 bf16 bytes from the staging slot, and
//                writes 32 E4M3 codes into the swizzled operand tile and the
//                scale byte into the slot's scale atom; then warps 2..5 (one
//                per TMEM lane quarter) copy the activation atom and both
//                weight atoms into the stage's scale columns; afterwards the
//                same warps drain the accumulator (64 columns each).
// Measured on that batched shape it is no faster than the quantise kernel
// followed by the CTA-pair GEMM (63.6 against 63.5 us), which is why the
// automatic path does not take it: a timing copy whose quantiser skips its
// loads and conversion still takes ~51 us, so the copy stream of this tiling
// (128-row boxes of 256 bytes from bf16 rows 14 KB apart, each weight tile
// read by four CTAs, ~3.6 TB/s) bounds it, not the quantiser (8 or 16
// quantiser warps measured the same).
// Every wait is bounded (on expiry the kernel records MXFP8_ERR_TIMEOUT and
// returns); no named barrier is used, so an expired wait cannot strand a warp.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

namespace mx {

namespace {

constexpr int FBM = 128;                   // rows per tile (MMA M)
constexpr int FBN = 256;                   // output columns per tile (MMA N)
constexpr int FBK = 128;                   // K elements per stage
constexpr int FSTAGES = 3;                 // operand ring: activation codes + weights
constexpr int FXSTAGES = 2;                // bf16 staging ring
constexpr int F_A_BYTES = FBM * FBK;       // 16 KB of codes
constexpr int F_B_BYTES = FBN * FBK;       // 32 KB of weights
constexpr int F_X_BOX = FBM * 128;         // one 128-row x 64-column bf16 box
constexpr int F_X_BYTES = 2 * F_X_BOX;     // a K tile of x: 32 KB
constexpr int F_Q_WARPS = 16;
constexpr int F_Q_THREADS = F_Q_WARPS * 32;
constexpr int F_THREADS = 64 + F_Q_THREADS;
constexpr int F_EPI_COLS = FBN / (F_Q_WARPS / 4);  // 64 accumulator columns per epilogue thread
constexpr int F_OFF_X = 0;
constexpr int F_OFF_A = F_OFF_X + FXSTAGES * F_X_BYTES;
constexpr int F_OFF_B = F_OFF_A + FSTAGES * F_A_BYTES;
constexpr int F_OFF_SFA = F_OFF_B + FSTAGES * F_B_BYTES;        // activation scale atom per stage
constexpr int F_OFF_SFB = F_OFF_SFA + FSTAGES * kAtomBytes;     // two weight scale atoms per stage
constexpr int F_OFF_BIAS = F_OFF_SFB + FSTAGES * 2 * kAtomBytes;  // per epilogue warp: its bias values
constexpr int F_OFF_BAR = F_OFF_BIAS + F_Q_WARPS * F_EPI_COLS * 2;
// per staging slot: x_full, x_empty; per operand slot: full (weights), empty
// (MMA done), atom_ready (codes + activation atom written), a_ready (scales
// in TMEM); then acc_full
constexpr int F_NUM_BARS = 2 * FXSTAGES + 4 * FSTAGES + 1;
constexpr int F_OFF_MISC = F_OFF_BAR + F_NUM_BARS * 8;
constexpr int F_SMEM_USED = F_OFF_MISC + 16;
constexpr int F_SMEM_ALLOC = F_SMEM_USED + 1024;
constexpr int F_T_ACC = 0;
constexpr int F_T_SFA = FBN;
constexpr int F_T_SFB = F_T_SFA + FSTAGES * 4;
constexpr int F_T_END = F_T_SFB + FSTAGES * 8;
constexpr int F_TMEM_COLS = 512;
// columns the epilogue's warm-up pass reads (allocated, never written)
constexpr int F_T_WARM = F_TMEM_COLS - F_EPI_COLS;
static_assert(F_T_END <= F_T_WARM, "tensor memory: the warm-up columns must be unused");
static_assert(F_SMEM_ALLOC <= 232448, "shared memory overflow");
static_assert(F_Q_THREADS == FBM * (FBK / 32), "one 32-element block per quantiser thread and K tile");
static_assert(F_EPI_COLS % 32 == 0, "epilogue chunks");

struct FArgs {
  const uint8_t* sfb;          // packed weight scale atoms
  const __nv_bfloat16* bias;   // [N] or nullptr
  __nv_bfloat16* out;          // [B, M, N]
  int B, M, N, K;
  int MT, NT, KT;              // tiles along M (128) and N (256), K tiles (128)
  int RTB;                     // 128-row atom tiles of the weights
  int wfmt;                    // weight (B operand) element format
};

__global__ void __launch_bounds__(F_THREADS, 1)
    gemm_fq_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const FArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* x_full = reinterpret_cast<uint64_t*>(smem + F_OFF_BAR);
  uint64_t* x_empty = x_full + FXSTAGES;
  uint64_t* full = x_empty + FXSTAGES;
  uint64_t* empty = full + FSTAGES;
  uint64_t* atom_ready = empty + FSTAGES;
  uint64_t* a_ready = atom_ready + FSTAGES;
  uint64_t* acc_full = a_ready + FSTAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + F_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + F_OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // one output tile per CTA: batch b, row tile mt, column tile nt
  const int per_b = a.MT * a.NT;
  const int b = blockIdx.x / per_b;
  const int nt = (blockIdx.x - b * per_b) / a.MT;
  const int mt = blockIdx.x - b * per_b - nt * a.MT;
  const int KT = a.KT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FXSTAGES; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], F_Q_WARPS);
    }
    for (int s = 0; s < FSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&atom_ready[s], F_Q_WARPS);
      mbar_init(&a_ready[s], 4);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, F_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int nb_atoms = min(2, a.RTB - nt * 2);
      const uint32_t w_tx = weight_tile_tx_bytes(FBN, a.wfmt) + nb_atoms * kAtomBytes;
      auto issue_w = [&](int k) {
        const int s = k % FSTAGES;
        mbar_arrive_expect_tx(&full[s], w_tx);
        tma_load_3d(smem + F_OFF_B + s * F_B_BYTES, &tmW, &full[s], k * FBK, nt * FBN, b);
        bulk_load(smem + F_OFF_SFB + s * 2 * kAtomBytes,
                  a.sfb + ((static_cast<int64_t>(b) * KT + k) * a.RTB + static_cast<int64_t>(nt) * 2) * kAtomBytes,
                  nb_atoms * kAtomBytes, &full[s]);
      };
      const int P0 = min(FSTAGES, KT);
      for (int k = 0; k < P0; ++k) issue_w(k);  // all slots are free at the start
      grid_dependency_wait();                   // x is the previous kernel's output
      int issued_x = 0, issued_w = P0;
      bool ok = true;
      for (int k = 0; k < KT; ++k) {
        const int xs = k % FXSTAGES;
        if (!mbar_wait(&x_empty[xs], ((k / FXSTAGES) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&x_full[xs], F_X_BYTES);
        uint8_t* dst = smem + F_OFF_X + xs * F_X_BYTES;
        tma_load_3d(dst, &tmX, &x_full[xs], k * FBK, mt * FBM, b);
        tma_load_3d(dst + F_X_BOX, &tmX, &x_full[xs], k * FBK + 64, mt * FBM, b);
        ++issued_x;
        if (k >= P0) {
          const int s = k % FSTAGES;
          if (!mbar_wait(&empty[s], ((k / FSTAGES) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          issue_w(k);
          ++issued_w;
        }
      }
      if (!ok) {
        // let every copy this thread started land before the CTA can exit
        for (int s = 0; s < FXSTAGES; ++s) {
          if (issued_x <= s) continue;
          const int last = ((issued_x - 1 - s) / FXSTAGES) * FXSTAGES + s;
          mbar_wait(&x_full[s], static_cast<uint32_t>((last / FXSTAGES) & 1), nullptr);
        }
        for (int s = 0; s < FSTAGES; ++s) {
          if (issued_w <= s) continue;
          const int last = ((issued_w - 1 - s) / FSTAGES) * FSTAGES + s;
          mbar_wait(&full[s], static_cast<uint32_t>((last / FSTAGES) & 1), nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc0 = idesc_with_types(idesc_mxf8(FBM, FBN), kFmtE4M3, a.wfmt);
      bool ok = true;
      for (int k = 0; k < KT; ++k) {
        const int s = k % FSTAGES;
        const uint32_t par = (k / FSTAGES) & 1;
        if (!mbar_wait(&full[s], par, abort_flag) || !mbar_wait(&a_ready[s], par, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(smem + F_OFF_A + s * F_A_BYTES));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(smem + F_OFF_B + s * F_B_BYTES));
        const uint32_t t_sfa = tmem + F_T_SFA + s * 4;
        const uint32_t t_sfb = tmem + F_T_SFB + s * 8;
#pragma unroll
        for (int kk = 0; kk < FBK / 32; ++kk)
          tc_mma_mxf8(tmem + F_T_ACC, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc0, kk, kk), t_sfa, t_sfb,
                      (k | kk) != 0);
        tc_commit(&empty[s]);
      }
      if (ok) tc_commit(acc_full);
      else __nanosleep(200000);  // let issued tensor-core work retire
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ quantiser, then epilogue
    const int qw = warp - 2;             // 0 .. F_Q_WARPS - 1
    const int quad = warp & 3;           // TMEM lane quarter this warp may access
    const int t = threadIdx.x - 64;
    const int r = t & (FBM - 1);         // tile row
    const int j = t >> 7;                // this thread's block of the K tile
    const int col0 = (qw >> 2) * F_EPI_COLS;
    uint4* bias_s = reinterpret_cast<uint4*>(smem + F_OFF_BIAS + qw * F_EPI_COLS * 2);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);

    // The bias may be read before the dependency wait (it is a weight-side
    // input), so it goes to shared memory now.
    if (a.bias != nullptr && lane < F_EPI_COLS / 8) {
      const int n = nt * FBN + col0 + 8 * lane;
      bias_s[lane] = n < a.N ? *reinterpret_cast<const uint4*>(a.bias + n) : make_uint4(0, 0, 0, 0);
    }
    __syncwarp();

    bool ok = true;
    for (int k = 0; k < KT; ++k) {
      const int xs = k % FXSTAGES, s = k % FSTAGES;
      const uint32_t xpar = (k / FXSTAGES) & 1, par = (k / FSTAGES) & 1;
      ok = ok && mbar_wait(&x_full[xs], xpar, abort_flag);
      uint4 v[4];
      if (ok) {
        // block j is 16-byte chunks 4 (j % 2) .. +3 of row r in box j / 2,
        // chunk c stored at c ^ (r % 8) (128-byte swizzle)
        const uint8_t* xrow = smem + F_OFF_X + xs * F_X_BYTES + (j >> 1) * F_X_BOX + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = *reinterpret_cast<const uint4*>(xrow + ((((j & 1) * 4 + q) ^ (r & 7)) << 4));
      }
      // the operand slot (codes, activation atom, TMEM scale columns) is free
      // once the MMAs of K tile k - FSTAGES are done
      ok = ok && mbar_wait(&empty[s], par ^ 1u, abort_flag);
      if (ok) {
        uint8_t* arow = smem + F_OFF_A + s * F_A_BYTES + r * 128;
        uint4 c0, c1;
        const uint32_t sbyte = quantize_block32(v, c0, c1);
        *reinterpret_cast<uint4*>(arow + (((2 * j) ^ (r & 7)) << 4)) = c0;
        *reinterpret_cast<uint4*>(arow + (((2 * j + 1) ^ (r & 7)) << 4)) = c1;
        smem[F_OFF_SFA + s * kAtomBytes + (r & 31) * 16 + (r >> 5) * 4 + j] = static_cast<uint8_t>(sbyte);
        fence_proxy_async_smem();  // the codes are read by the tensor cores
      }
      __syncwarp();
      if (lane == 0 && ok) {
        // the staging slot is released only here, after the quantiser has
        // consumed the values it loaded (a release right after the loads was
        // measured no faster and once produced wrong bytes)
        mbar_arrive(&x_empty[xs]);
        mbar_arrive(&atom_ready[s]);
      }
      if (qw < 4) {
        // one warp per TMEM lane quarter: atom line `lane` (rows lane + 32 i,
        // 4 blocks each) of the activation atom and of both weight atoms into
        // this quarter's lanes of the stage's scale columns (the MMA reads
        // them from every quarter)
        ok = ok && mbar_wait(&atom_ready[s], par, abort_flag) && mbar_wait(&full[s], par, abort_flag);
        if (ok) {
          const uint4 va = *reinterpret_cast<const uint4*>(smem + F_OFF_SFA + s * kAtomBytes + lane * 16);
          const uint4 vb0 = *reinterpret_cast<const uint4*>(smem + F_OFF_SFB + s * 2 * kAtomBytes + lane * 16);
          const uint4 vb1 =
              *reinterpret_cast<const uint4*>(smem + F_OFF_SFB + s * 2 * kAtomBytes + kAtomBytes + lane * 16);
          tmem_st_32x32b_x4(lane_base + F_T_SFA + s * 4, va.x, va.y, va.z, va.w);
          tmem_st_32x32b_x4(lane_base + F_T_SFB + s * 8, vb0.x, vb0.y, vb0.z, vb0.w);
          tmem_st_32x32b_x4(lane_base + F_T_SFB + s * 8 + 4, vb1.x, vb1.y, vb1.z, vb1.w);
          tmem_st_wait();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&a_ready[s]);
      }
    }

    // ------------------------------------------------------------ epilogue
    // The first pass (live == false) is a warm-up of the drain and store code
    // on tensor-memory columns nothing writes, with the wait and the stores
    // skipped (see gemm.cu); here it runs after the main loop, while the last
    // MMAs are still in the tensor pipe.  The pass count starts from an opaque
    // register so that one copy of the body serves both passes.
    int pass;
    asm volatile("mov.s32 %0, -1;" : "=r"(pass));
    for (; pass <= 0; ++pass) {
      const bool live = pass >= 0;
      if (live) {
        ok = ok && mbar_wait(acc_full, 0, abort_flag);
        if (!ok) break;
        tc_fence_after();
      }
      const int row = mt * FBM + quad * 32 + lane;
      const uint32_t taddr = lane_base + (live ? F_T_ACC + col0 : F_T_WARM);
      __nv_bfloat16* orow = a.out + (static_cast<int64_t>(b) * a.M + row) * a.N;
#pragma unroll
      for (int c = 0; c < F_EPI_COLS / 32; ++c) {
        uint32_t rr[32];
        tmem_ld_32x32b_x32(taddr + c * 32, rr);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float bv[8];
          if (a.bias != nullptr) {
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
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[8 * g + 2 * i]) + bv[2 * i],
                                __uint_as_float(rr[8 * g + 2 * i + 1]) + bv[2 * i + 1]);
          // 8 outputs per 16-byte store (N % 8 == 0); rows / columns past M, N are not written
          const int n = nt * FBN + col0 + c * 32 + 8 * g;
          if (live && row < a.M && n < a.N)
            *reinterpret_cast<uint4*>(orow + n) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, F_TMEM_COLS);
  }
}

// 3-D map over bf16 x [B][M][K], box {64 columns, 128 rows, 1}, 128-byte
// swizzle, zero fill outside the tensor (ragged M reads zero rows).
cudaError_t make_x_bf16_map(CUtensorMap* map, const void* x, int64_t B, int64_t M, int64_t K, const char** msg) {
  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) {
    *msg = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K * 2), static_cast<cuuint64_t>(M * K * 2)};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(FBM), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected the bf16 activations";
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace

int64_t fused_quantize_tiles(int64_t B, int64_t M, int64_t N) {
  return B * ceil_div(M, FBM) * ceil_div(N, FBN);
}

cudaError_t launch_gemm_fq(const FusedProblem& p, int sms, cudaStream_t stream, const char** msg) {
  const int64_t tiles = fused_quantize_tiles(p.B, p.M, p.N);
  if (tiles < 1 || tiles > sms || p.N % 8 != 0 || p.K % FBK != 0) {
    *msg = "fused-quantise GEMM: shape outside its range";
    return cudaErrorInvalidValue;
  }
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM_ALLOC);
    if (e != cudaSuccess) {
      *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return e;
    }
    attr_set[dev] = true;
  }
  CUtensorMap mx_, mw;
  cudaError_t e = make_x_bf16_map(&mx_, p.x, p.B, p.M, p.K, msg);
  if (e != cudaSuccess) return e;
  e = make_operand_map(&mw, p.w, p.B, p.N, p.K, FBN, msg, p.wfmt);
  if (e != cudaSuccess) return e;
  FArgs a;
  a.sfb = p.sfw;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.B = static_cast<int>(p.B);
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.MT = static_cast<int>(ceil_div(p.M, FBM));
  a.NT = static_cast<int>(ceil_div(p.N, FBN));
  a.KT = static_cast<int>(p.K / FBK);
  a.RTB = static_cast<int>(ceil_div(p.N, kAtomRows));
  a.wfmt = p.wfmt;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles), 1, 1);
  cfg.blockDim = dim3(F_THREADS, 1, 1);
  cfg.dynamicSmemBytes = F_SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_fq_kernel, mx_, mw, a);
  if (e != cudaSuccess) *msg = "fused-quantise GEMM launch failed";
  return e;
}

cudaError_t take_status_fq(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
