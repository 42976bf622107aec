// gemm_pair.cu - the block-scaled MXFP8 GEMM on CTA pairs (cta_group::2).
//
// Same function as gemm.cu (the block-scaled product and bias add of
// "AiterFlyDSLMxfp8LinearKernel.apply_weights", aiter_flydsl page, batched per
// "Mxfp8LinearLayerConfig.bmm_batch_size"), for M > 128.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2: CTA r holds rows [128 r, 128 r + 128) of the
// activation tile and rows [128 r, 128 r + 128) of the 256-row weight tile in
// its shared memory, and receives the 128 x 256 fp32 accumulator of its rows
// in its tensor memory.  Per SM and K tile that is 16 KB of activations and
// 16 KB of weights for the work that takes 16 + 32 KB with one CTA per tile,
// and one MMA instruction covers 256 rows: each block-scaled MMA has a large
// fixed cost, so the widest shape per instruction is the fastest.
//
// The kernel is launched with programmatic stream serialization: the first
// ring round of weight tiles is issued before griddepcontrol.wait, the
// activation tiles and scales (the previous kernel's output) after it.
//
// Warp roles per CTA (both CTAs run every role but the MMA issuer):
//   warp 0       TMA producer for this CTA's operand halves; both CTAs' copies
//                complete on the even CTA's `full` barrier, whose transaction
//                count the even CTA alone posts (for both), so the odd CTA
//                sends no barrier traffic of its own;
//   warp 1       TMEM allocation (collective over the pair); in the even CTA
//                one lane issues the pair MMAs and commits them to the
//                barriers of both CTAs (multicast);
//   warps 2..5   scale-factor writers: read this CTA's activation scale atom
//                and both weight scale atoms straight from global memory a few
//                K tiles ahead, and once a pair of stages is free tcgen05.st
//                them (all 256 weight columns, in order: each CTA's half of
//                the pair MMA reads the scales from its own tensor memory),
//                then arrive on the even CTA's sf_ready barrier of the pair
//                (the even CTA's writers first wait for both stages' operands,
//                so the MMA issuer waits once per two stages);
//   warps 6..13  epilogue: drain this CTA's accumulator as bf16, arrive on the
//                even CTA's acc_empty barrier, TMA-store the rows (and, for the
//                MXFP8 hand-off, their E4M3 codes through the same staging box:
//                per-row 16-byte stores of the codes measured 4-8 us slower
//                at MLP-up).
// One thread issuing every copy of a stage is the first limit here (a TMA or
// bulk-copy issue costs ~100-150 cycles, a stage of MMAs ~550), which is why
// the scale atoms do not go through the producer.  Every wait is bounded; a
// cluster barrier at the start (barrier initialisation) and at the end (before
// deallocation) is reached on every path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_epilogue.cuh"
#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

namespace mx {

namespace {

constexpr int PBM = 128;    // activation rows per CTA (256 per pair)
constexpr int PBK = 128;    // K elements per stage
constexpr int PBN = 256;    // output columns per pair tile; each CTA loads PBN / 2 weight rows
constexpr int PSTAGES = 6;
constexpr int P_A_BYTES = PBM * PBK;
constexpr int P_B_BYTES = (PBN / 2) * PBK;
constexpr int P_SF_WARPS = 4;
constexpr int P_SF_AHEAD = 2;  // stage pairs of scale atoms each writer holds in registers
constexpr int P_EPI_WARPS = 8;
constexpr int P_EPI_THREADS = P_EPI_WARPS * 32;
constexpr int P_EPI_COLS = PBN / (P_EPI_WARPS / 4);
constexpr int P_STAGE_OUT = 32 * 32 * 2;
constexpr int P_THREADS = 64 + P_SF_WARPS * 32 + P_EPI_THREADS;
constexpr int P_OFF_A = 0;
constexpr int P_OFF_B = P_OFF_A + PSTAGES * P_A_BYTES;
constexpr int P_OFF_OUT = P_OFF_B + PSTAGES * P_B_BYTES;
constexpr int P_OFF_BIAS = P_OFF_OUT + P_EPI_WARPS * P_STAGE_OUT;  // per epilogue warp: its 128 bias values
constexpr int P_OFF_BAR = P_OFF_BIAS + P_EPI_WARPS * P_EPI_COLS * 2;
// per stage: full (operands of both CTAs, in the even CTA) and empty; per
// stage pair: sf_ready (in the even CTA); then acc_full, acc_empty
constexpr int P_NUM_BARS = 2 * PSTAGES + PSTAGES / 2 + 2;
constexpr int P_OFF_MISC = P_OFF_BAR + P_NUM_BARS * 8;
constexpr int P_SMEM_USED = P_OFF_MISC + 16;
constexpr int P_SMEM_ALLOC = P_SMEM_USED + 1024;
constexpr int P_T_ACC = 0;
constexpr int P_T_SFA = PBN;
constexpr int P_T_SFB = P_T_SFA + PSTAGES * 4;
constexpr int P_T_END = P_T_SFB + PSTAGES * 8;
constexpr int P_TMEM_COLS = 512;
// columns the epilogue's warm-up pass reads (allocated, never written)
constexpr int P_T_WARM = P_TMEM_COLS - P_EPI_COLS;
static_assert(P_T_END <= P_TMEM_COLS, "tensor memory overflow");
static_assert(P_T_WARM >= P_T_END, "the warm-up columns must be unused");
static_assert(P_SMEM_ALLOC <= 232448, "shared memory overflow");
static_assert(PSTAGES % 2 == 0, "scale factors are written per pair of stages");
static_assert(P_EPI_COLS == 128, "the MXFP8 hand-off quantises 128 columns (one scale word) per thread");

struct PArgs {
  const uint8_t* sfa;  // activation scales: packed atoms, or row-major [B, M, K/32] when sfa_rowmajor
  const uint8_t* sfb;
  const __nv_bfloat16* bias;
  uint8_t* yq;   // MXFP8 hand-off outputs (nullptr: none), see mx_epilogue.cuh
  uint8_t* ysf;
  int B, M, N, K;
  int MT2, NT, KT;  // 256-row pair tiles, 256-column tiles, K tiles
  int RTA, RTB;     // 128-row atom tiles of A and of W
  int RTY, KTY;     // atom tiles of the hand-off scales (rows, K tiles = N / 128)
  int store_bf16;   // 0: the bf16 output is not written
  int wfmt;         // weight (B operand) element format
  int total_tiles;
  int splits;       // K splits per tile (split-K): > 1 writes fp32 partials through tmPart
  int units;        // total_tiles * splits
  int sfa_rowmajor; // 1: sfa is the caller's row-major x_scale (no repack kernel before this one)
  int n_fast;       // tile order: 1 = column tiles vary fastest, 0 = row tiles
};

__device__ __forceinline__ void pair_tile_coords(int tile, const PArgs& a, int& b, int& mt2, int& nt) {
  const int per_b = a.MT2 * a.NT;
  b = tile / per_b;
  const int t = tile - b * per_b;
  if (a.n_fast) {
    mt2 = t / a.NT;
    nt = t - mt2 * a.NT;
  } else {
    nt = t / a.MT2;
    mt2 = t - nt * a.MT2;
  }
}

// Work unit u = tile * splits + s: output tile `tile`, K tiles [kt_lo, kt_hi)
// (the splits of one tile go to consecutive pairs, which run them at once).
__device__ __forceinline__ void unit_coords(int u, const PArgs& a, int& b, int& mt2, int& nt, int& s, int& kt_lo,
                                            int& kt_hi) {
  const int tile = u / a.splits;
  s = u - tile * a.splits;
  pair_tile_coords(tile, a, b, mt2, nt);
  kt_lo = s * a.KT / a.splits;
  kt_hi = (s + 1) * a.KT / a.splits;
}

// K steps (stages) of all units pair `pair` runs.
__device__ __forceinline__ int64_t pair_steps(int pair, int npairs, const PArgs& a) {
  int64_t n = 0;
  for (int u = pair; u < a.units; u += npairs) {
    const int s = u % a.splits;
    n += (s + 1) * a.KT / a.splits - s * a.KT / a.splits;
  }
  return n;
}

__global__ void __launch_bounds__(P_THREADS, 1)
    gemm_mxf8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmPart,
                          const __grid_constant__ CUtensorMap tmYq,
                          const PArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_OFF_BAR);
  uint64_t* empty = full + PSTAGES;
  uint64_t* sf_ready = empty + PSTAGES;  // one per stage pair
  uint64_t* acc_full = sf_ready + PSTAGES / 2;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P_OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P_OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;  // clusters are (2, 1, 1)
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);                        // the even CTA's producer (even CTA's copy is used)
      mbar_init(&empty[s], 1);                       // the even CTA's commit
    }
    for (int s = 0; s < PSTAGES / 2; ++s)
      mbar_init(&sf_ready[s], 2 * P_SF_WARPS);       // one arrive per writer warp of both CTAs
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * P_EPI_WARPS);           // one arrive per epilogue warp of both CTAs
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmOut);
    if (args.splits > 1) prefetch_tmap(&tmPart);
    if (args.yq != nullptr) prefetch_tmap(&tmYq);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anyone arrives remotely
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // With split K the next kernel is this call's reduce, which reads the
  // partials only after its own dependency wait: let it launch now.
  if (args.splits > 1 && threadIdx.x == 0) launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Prologue for the first ring round (all slots free): the weight tiles
      // do not depend on the kernel before this one in the stream, the
      // activation tiles (its output) do.  Issue the weights, wait for the
      // dependency (programmatic dependent launch), then the activations.
      const int P0 = static_cast<int>(min(static_cast<int64_t>(PSTAGES), pair_steps(pair, npairs, args)));
      for (int pass = 0; pass < 2; ++pass) {
        int u = pair, kt = 0, kt_hi = 0, b = 0, mt2 = 0, nt = 0, sp = 0;
        if (P0 > 0) unit_coords(u, args, b, mt2, nt, sp, kt, kt_hi);
        for (int s0 = 0; s0 < P0; ++s0) {
          const uint32_t full_even = map_shared_rank(smem_u32(&full[s0]), 0);
          if (pass == 0) {
            if (leader) mbar_arrive_expect_tx(&full[s0], 2 * (P_A_BYTES + weight_tile_tx_bytes(PBN / 2, args.wfmt)));
            tma_load_3d_cluster_bar(smem + P_OFF_B + s0 * P_B_BYTES, &tmB, full_even, kt * PBK,
                                    nt * PBN + static_cast<int>(rank) * (PBN / 2), b);
          } else {
            tma_load_3d_cluster_bar(smem + P_OFF_A + s0 * P_A_BYTES, &tmA, full_even, kt * PBK,
                                    (mt2 * 2 + static_cast<int>(rank)) * PBM, b);
          }
          if (++kt == kt_hi) {
            u += npairs;
            if (u < args.units) unit_coords(u, args, b, mt2, nt, sp, kt, kt_hi);
          }
        }
        if (pass == 0) grid_dependency_wait();
      }
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = pair; ok && u < args.units; u += npairs) {
        int b, mt2, nt, sp, kt_lo, kt_hi;
        unit_coords(u, args, b, mt2, nt, sp, kt_lo, kt_hi);
        const int rt_a = mt2 * 2 + static_cast<int>(rank);  // this CTA's activation row tile
        for (int kt = kt_lo; kt < kt_hi; ++kt) {
          if (issued < P0) {  // issued by the prologue
            ++issued;
            if (++stage == PSTAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // Both CTAs' copies complete on the even CTA's barrier.  The odd
          // CTA's bytes may land before the even CTA posts the count (the
          // transaction count goes negative for a while); they cannot land a
          // phase early, because this stage was freed by a commit that
          // followed the MMA that waited for the barrier's previous phase.
          const uint32_t full_even = map_shared_rank(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (P_A_BYTES + weight_tile_tx_bytes(PBN / 2, args.wfmt)));
          tma_load_3d_cluster_bar(smem + P_OFF_A + stage * P_A_BYTES, &tmA, full_even, kt * PBK, rt_a * PBM, b);
          tma_load_3d_cluster_bar(smem + P_OFF_B + stage * P_B_BYTES, &tmB, full_even, kt * PBK,
                                  nt * PBN + static_cast<int>(rank) * (PBN / 2), b);
          ++issued;
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every commit the even CTA sends to this CTA's empty barriers must have
      // arrived before exit; the last commit of a stage follows the MMA that
      // waited for its operands, so the copies have landed too.
      for (int s = 0; s < PSTAGES; ++s) {
        if (issued <= s) continue;
        const int64_t last = ((issued - 1 - s) / PSTAGES) * PSTAGES + s;
        const uint32_t par = static_cast<uint32_t>((last / PSTAGES) & 1);
        mbar_wait(&empty[s], par, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t idesc0 = idesc_with_types(idesc_mxf8(2 * PBM, PBN), kFmtE4M3, args.wfmt);
      for (int u = pair; ok && u < args.units; u += npairs) {
        const int sp = u % args.splits;
        const int kt_lo = sp * args.KT / args.splits, kt_hi = (sp + 1) * args.KT / args.splits;
        if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = kt_lo; kt < kt_hi; ++kt) {
          // operands of both CTAs landed, and both CTAs' scales are in TMEM
          // one wait per pair of stages: the even CTA's scale writers arrive on
          // sf_ready only after both stages' operands have landed
          if ((stage & 1) == 0 && !mbar_wait(&sf_ready[stage >> 1], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(smem + P_OFF_A + stage * P_A_BYTES));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(smem + P_OFF_B + stage * P_B_BYTES));
          const uint32_t t_sfa = tmem + P_T_SFA + stage * 4;
          const uint32_t t_sfb = tmem + P_T_SFB + stage * 8;
#pragma unroll
          for (int kk = 0; kk < PBK / 32; ++kk)
            tc_mma_mxf8_pair(tmem + P_T_ACC, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc0, kk, kk),
                             t_sfa, t_sfb, ((kt - kt_lo) | kk) != 0);
          tc_commit_pair_multicast(&empty[stage], 0x3);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(acc_full, 0x3);
        acc_phase ^= 1u;
      }
      if (!ok) __nanosleep(200000);  // let issued tensor-core work retire
    }
    __syncwarp();
  } else if (warp < 2 + P_SF_WARPS) {
    // ------------------------------------------------------------ scale-factor writers
    // Each writer warp owns TMEM lanes [32 (warp % 4), +32) and writes the
    // same atom lines there (one 16-byte line per lane and atom).  Each K
    // tile's atoms are fetched P_SF_AHEAD K tiles before they are written; the
    // write waits for the stage's previous MMAs (empty barrier).
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t ready_even = map_shared_rank(smem_u32(sf_ready), 0);
    grid_dependency_wait();  // the activation scales are the previous kernel's output
    const int64_t total = pair_steps(pair, npairs, args);
    // Fetch cursor: pointers to this lane's line of the activation atom and
    // of the first weight atom of K tile f_kt of unit f_u; advancing a K
    // tile adds one K-tile row of atoms.
    // With row-major activation scales the lane gathers its atom line itself:
    // word i of line `lane` is the 4 scale bytes (blocks 4 kt .. 4 kt + 3) of
    // tile row lane + 32 i, i.e. 4 aligned bytes of that row (K % 128 == 0);
    // rows past M read as 0 (their outputs are never stored).
    int f_u = pair, f_kt = 0, f_kt_hi = 0;
    const uint8_t* f_a = nullptr;
    const uint8_t* f_w = nullptr;
    bool f_has_a = false, f_has_w1 = false;
    uint32_t f_rows = 0;  // row-major mode: bit i set when row lane + 32 i is < M
    const int64_t kb = args.K / 32;
    const int64_t a_step = args.sfa_rowmajor ? 4 : static_cast<int64_t>(args.RTA) * kAtomBytes;
    const int64_t w_step = static_cast<int64_t>(args.RTB) * kAtomBytes;
    auto start_tile = [&]() {
      if (f_u >= args.units) return;
      int b, mt2, nt, sp;
      unit_coords(f_u, args, b, mt2, nt, sp, f_kt, f_kt_hi);
      const int rt_a = mt2 * 2 + static_cast<int>(rank);
      const int64_t arow = static_cast<int64_t>(b) * args.KT + f_kt;
      f_has_a = rt_a < args.RTA;
      f_has_w1 = 2 * nt + 1 < args.RTB;
      if (args.sfa_rowmajor) {
        const int r0 = rt_a * kAtomRows + lane;
        f_rows = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) f_rows |= (r0 + 32 * i < args.M ? 1u : 0u) << i;
        f_a = args.sfa + (static_cast<int64_t>(b) * args.M + (f_rows & 1u ? r0 : 0)) * kb + 4 * f_kt;
      } else {
        f_a = args.sfa + (arow * args.RTA + (f_has_a ? rt_a : 0)) * kAtomBytes + lane * 16;
      }
      f_w = args.sfb + (arow * args.RTB + 2 * nt) * kAtomBytes + lane * 16;
    };
    start_tile();
    auto fetch = [&](uint4& va, uint4& vb0, uint4& vb1) {
      const uint4 zero = make_uint4(0, 0, 0, 0);
      if (args.sfa_rowmajor) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = (f_rows >> i) & 1u ? __ldg(reinterpret_cast<const uint32_t*>(f_a + 32 * i * kb)) : 0u;
        va = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        va = f_has_a ? __ldg(reinterpret_cast<const uint4*>(f_a)) : zero;
      }
      vb0 = __ldg(reinterpret_cast<const uint4*>(f_w));
      vb1 = f_has_w1 ? __ldg(reinterpret_cast<const uint4*>(f_w + kAtomBytes)) : zero;
      f_a += a_step;
      f_w += w_step;
      if (++f_kt == f_kt_hi) {
        f_u += npairs;
        start_tile();
      }
    };
    // Stages go in pairs (2i, 2i + 1), which share a round of the ring.  The
    // MMAs finish in issue order, so once the second stage's previous MMAs
    // are done (its empty barrier) both scale slots are free; one arrive on
    // sf_ready[i] then publishes both.  A lone last stage waits on its own.
    uint4 ra[2 * P_SF_AHEAD], rb0[2 * P_SF_AHEAD], rb1[2 * P_SF_AHEAD];
#pragma unroll
    for (int d = 0; d < 2 * P_SF_AHEAD; ++d)
      if (d < total) fetch(ra[d], rb0[d], rb1[d]);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t j0 = 0; ok && j0 < total; j0 += 2 * P_SF_AHEAD) {
#pragma unroll
      for (int d = 0; d < 2 * P_SF_AHEAD; d += 2) {
        const int64_t j = j0 + d;
        if (!ok || j >= total) break;
        const bool two = j + 1 < total;
        if (!mbar_wait(&empty[stage + (two ? 1 : 0)], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read these scale slots are done
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int sl = stage + h;
          tmem_st_32x32b_x4(lane_base + P_T_SFA + sl * 4, ra[d + h].x, ra[d + h].y, ra[d + h].z, ra[d + h].w);
          tmem_st_32x32b_x4(lane_base + P_T_SFB + sl * 8, rb0[d + h].x, rb0[d + h].y, rb0[d + h].z, rb0[d + h].w);
          tmem_st_32x32b_x4(lane_base + P_T_SFB + sl * 8 + 4, rb1[d + h].x, rb1[d + h].y, rb1[d + h].z,
                            rb1[d + h].w);
        }
        tmem_st_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (j + h + 2 * P_SF_AHEAD < total) fetch(ra[d + h], rb0[d + h], rb1[d + h]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) {
            // the operands of both stages (both CTAs' copies complete here)
            bool landed = mbar_wait(&full[stage], phase, abort_flag);
            if (landed && two) landed = mbar_wait(&full[stage + 1], phase, abort_flag);
            if (landed) mbar_arrive(&sf_ready[stage >> 1]);
          } else
            mbar_arrive_remote(ready_even + static_cast<uint32_t>((stage >> 1) * 8));
        }
        stage += 2;
        if (stage == PSTAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2 - P_SF_WARPS;
    const int quad = warp & 3;
    const int col0 = (ew >> 2) * P_EPI_COLS;
    uint8_t* stage_out = smem + P_OFF_OUT + ew * P_STAGE_OUT;
    uint4* bias_s = reinterpret_cast<uint4*>(smem + P_OFF_BIAS + ew * P_EPI_COLS * 2);
    const uint32_t acc_empty_even = map_shared_rank(smem_u32(acc_empty), 0);
    uint32_t acc_phase = 0;
    bool pending = false;
    // The first pass (live == false) is a warm-up: it runs the drain and
    // store code below once, on tensor-memory columns nothing writes, with
    // every wait, arrive and global write skipped.  Its only effect is that
    // this code is in the SM's instruction cache when the first accumulator
    // is ready; without it the first tile's drain took ~1.6-1.9 us instead of
    // ~0.4 us, at the same moment on every SM (their fetches of the code
    // from DRAM merge), and a one-tile call's stores ~2 us.  The pass count
    // starts from an opaque register so that one copy of the body serves both.
    int pass;
    asm volatile("mov.s32 %0, -1;" : "=r"(pass));
    for (int u = pair; u < args.units; ++pass) {
      const bool live = pass >= 0;
      int b, mt2, nt, sp, kt_lo, kt_hi;
      unit_coords(u, args, b, mt2, nt, sp, kt_lo, kt_hi);
      if (live) u += npairs;
      if (live && args.bias != nullptr && args.splits == 1) {
        // this warp's 128 bias values (zero past N) into shared memory while
        // the tile's MMAs run, so that the drain below reads no global memory
        if (lane < P_EPI_COLS / 8) {
          const int n = nt * PBN + col0 + 8 * lane;
          bias_s[lane] = n < args.N ? *reinterpret_cast<const uint4*>(args.bias + n) : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      if (live) {
        if (!mbar_wait(acc_full, acc_phase, abort_flag)) break;
        tc_fence_after();
      }
      const int row0 = mt2 * 2 * PBM + static_cast<int>(rank) * PBM + quad * 32;
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(quad * 32) << 16) + (live ? P_T_ACC + col0 : P_T_WARM);
      if (args.splits > 1) {
        // split-K: this unit's fp32 partial, no bias, through 32-row x
        // 16-column boxes into the workspace [splits * B][M][N] at
        // z = split * B + b (rows / columns past M, N are clipped); the
        // reduce kernel adds the partials in split order
        for (int c = 0; c < P_EPI_COLS / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (lane == 0 && pending) bulk_wait_group_read0();
            __syncwarp();
            uint4* dst = reinterpret_cast<uint4*>(stage_out + lane * 64);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(r[16 * h + 4 * q], r[16 * h + 4 * q + 1], r[16 * h + 4 * q + 2],
                                  r[16 * h + 4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && live) {
              tma_store_3d(&tmPart, stage_out, nt * PBN + col0 + c * 32 + 16 * h, row0, sp * args.B + b);
              bulk_commit_group();
              pending = true;
            }
          }
        }
        if (live) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(acc_empty_even);
          acc_phase ^= 1u;
        }
        continue;
      }
      uint32_t packed[P_EPI_COLS / 2];
#pragma unroll
      for (int c = 0; c < P_EPI_COLS / 32; ++c) {
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
        if (lane == 0) mbar_arrive_remote(acc_empty_even);  // the even CTA may start the next tile
        acc_phase ^= 1u;
      }

      // the same bf16 values quantised for the next layer (MXFP8 hand-off)
      if (args.yq != nullptr) {
        // the same bf16 values quantised for the next layer: this lane's 128
        // codes go through the warp's staging box in two 64-column halves
        // (32 rows x 64 bytes each, TMA stores clip rows past M), the scale
        // word of its row straight to the packed atoms
        const int n0 = nt * PBN + col0;
        uint32_t sword = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 cq[4];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * h + cc;
            const uint4 v[4] = {make_uint4(packed[16 * c], packed[16 * c + 1], packed[16 * c + 2], packed[16 * c + 3]),
                                make_uint4(packed[16 * c + 4], packed[16 * c + 5], packed[16 * c + 6], packed[16 * c + 7]),
                                make_uint4(packed[16 * c + 8], packed[16 * c + 9], packed[16 * c + 10], packed[16 * c + 11]),
                                make_uint4(packed[16 * c + 12], packed[16 * c + 13], packed[16 * c + 14],
                                           packed[16 * c + 15])};
            sword |= quantize_block32(v, cq[2 * cc], cq[2 * cc + 1]) << (8 * c);
          }
          if (lane == 0 && pending) bulk_wait_group_read0();
          __syncwarp();
          uint4* dst = reinterpret_cast<uint4*>(stage_out + lane * 64);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = cq[q];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && live) {
            tma_store_3d(&tmYq, stage_out, n0 + 64 * h, row0, b);
            bulk_commit_group();
            pending = true;
          }
        }
        const int row = row0 + lane;
        if (live && row < args.M && n0 < args.N) {
          const int64_t atom = (static_cast<int64_t>(b) * args.KTY + n0 / kTileK) * args.RTY + (row >> 7);
          *reinterpret_cast<uint32_t*>(args.ysf + atom * kAtomBytes + (row & 31) * 16 + ((row >> 5) & 3) * 4) = sword;
        }
      }
      if (!args.store_bf16) continue;
#pragma unroll
      for (int c = 0; c < P_EPI_COLS / 32; ++c) {
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
          tma_store_3d(&tmOut, stage_out, nt * PBN + col0 + c * 32, row0, b);
          bulk_commit_group();
          pending = true;
        }
      }
    }
    if (lane == 0 && pending) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA of the pair leaves while the other may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmProblem& p, int sms, cudaStream_t stream, const char** msg) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_mxf8_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         P_SMEM_ALLOC);
    if (e != cudaSuccess) {
      *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return e;
    }
    attr_set[dev] = true;
  }
  CUtensorMap ma, mb, mo, mp, my;
  cudaError_t e = make_operand_map(&ma, p.a, p.B, p.M, p.K, PBM, msg);
  if (e != cudaSuccess) return e;
  e = make_operand_map(&mb, p.w, p.B, p.N, p.K, PBN / 2, msg, p.wfmt);
  if (e != cudaSuccess) return e;
  const int splits = p.part != nullptr && p.splits > 1 ? p.splits : 1;
  // without a bf16 output (hand-off only, or split-K partials) the map is never
  // used; any aligned address will do
  void* out_any = p.out != nullptr ? p.out : (p.yq != nullptr ? static_cast<void*>(p.yq) : static_cast<void*>(p.part));
  e = make_output_map(&mo, out_any, p.B, p.M, p.N, msg);
  if (e != cudaSuccess) return e;
  if (p.yq != nullptr) {
    // E4M3 codes [B][M][N], box {64 columns, 32 rows, 1}, no swizzle
    EncodeTiledFn encode = encode_tiled_fn();
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(p.B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M * p.N)};
    const cuuint32_t box[3] = {64, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode == nullptr ||
        encode(&my, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.yq, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS) {
      *msg = "cuTensorMapEncodeTiled rejected the hand-off codes";
      return cudaErrorInvalidValue;
    }
  } else {
    my = mo;  // unused
  }
  if (e != cudaSuccess) return e;
  if (splits > 1) {
    e = make_partial_map(&mp, p.part, static_cast<int64_t>(splits) * p.B, p.M, p.N, msg);
    if (e != cudaSuccess) return e;
  } else {
    mp = mo;  // unused
  }

  PArgs a;
  a.sfa = p.sfa;
  a.sfb = p.sfb;
  a.sfa_rowmajor = p.sfa_rowmajor;
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
  a.MT2 = static_cast<int>(ceil_div(p.M, 2 * PBM));
  a.NT = static_cast<int>(ceil_div(p.N, PBN));
  a.KT = static_cast<int>(p.K / PBK);
  a.RTA = static_cast<int>(ceil_div(p.M, kAtomRows));
  a.RTB = static_cast<int>(ceil_div(p.N, kAtomRows));
  a.total_tiles = a.B * a.MT2 * a.NT;
  a.splits = splits;
  a.units = a.total_tiles * splits;
  // The pairs of one round run consecutive tiles at once: sweep the operand
  // with fewer bytes fastest, so that it stays in L2 while each tile of the
  // larger one is read from DRAM once (M >= N: the weights stay resident;
  // at M = N, K = 14336 behind a hand-off this measured 347.5 -> 342.7 us
  // for the two-layer chain).
  a.n_fast = p.M >= p.N ? 1 : 0;
  // split-K: the partials carry no bias and no hand-off; the reduce adds them
  if (splits > 1) {
    a.bias = nullptr;
    a.yq = a.ysf = nullptr;
    a.store_bf16 = 0;
  }
  const int pairs = a.units < sms / 2 ? a.units : sms / 2;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(P_THREADS, 1, 1);
  cfg.dynamicSmemBytes = P_SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the prologue and the first weight tiles
  // overlap the end of the kernel before (normally the quantiser)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, gemm_mxf8_pair_kernel, ma, mb, mo, mp, my, a);
  if (e != cudaSuccess) {
    *msg = "pair GEMM launch failed";
    return e;
  }
  if (splits > 1) {
    e = launch_splitk_reduce(p.part, splits, p.B, p.M, p.N, p.bias, p.out, p.yq, p.ysf, sms, stream);
    if (e != cudaSuccess) *msg = "split-K reduce launch failed";
  }
  return e;
}

}  // namespace mx

namespace mx {

cudaError_t take_status_pair(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
