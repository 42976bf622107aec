// gemm_decode.cu - the small-M (decode) path of the MXFP8 linear layer.
//
// out[m, n] = bf16( sum_k deq(x)[m, k] * deq(w)[n, k] + bias[n] ), M <= 128,
// with x bf16 quantised to MXFP8 inside the kernel: the block-scaled product
// and bias add of "AiterFlyDSLMxfp8LinearKernel.apply_weights" (aiter_flydsl
// page), with its mxfp8_e4m3_quantize step fused into the GEMM producer.
//
// At small M the layer is bound by reading the weights once from HBM, so:
//   * the weights are the MMA's A operand (M = 128 weight rows per CTA) and the
//     tokens its B operand (N = 16, 32, 64 or 128 >= M), so no MMA rows are wasted
//     on padding tokens;
//   * K is split over a cluster of S CTAs (S in {1, 2, 4, 8}, the largest
//     whose clusters all fit on the GPU at once); each CTA streams its
//     128 x K/S weight slice through a TMA ring (at N = K = 4096: S = 4 -- at
//     one CTA per SM only 15 clusters of 8 fit at once -- so 8 K tiles per
//     CTA, which up to 16 tokens are all in flight from the start);
//   * warps 2..9 read x (bf16, from L2) and quantise it with the same device
//     function as the standalone quantize kernel (one lane per 32-element
//     block of the M real token rows), writing E4M3 codes straight into the
//     128-byte-swizzled operand tile and the scales into the scale-factor
//     atom.  They work on groups of K tiles and issue the next group's loads
//     before quantising the current one, so the latency of x is paid about
//     once.  A pre-quantised x (E4M3 codes and row-major scales, the
//     QuantizedActivation input of apply_weights) takes the same path with the
//     quantisation replaced by a copy of the block's 32 codes and scale byte;
//   * the S fp32 partial tiles meet in distributed shared memory: CTA r owns
//     weight rows [r*128/S, (r+1)*128/S); every CTA stores its partial for
//     those rows straight into the owner's receive buffer (remote shared-memory
//     stores), then one cluster barrier, then each owner sums its S partials
//     in the fixed order 0..S-1 (deterministic), adds the bias and stores bf16;
//     with S = 1 the epilogue warps store the output straight from TMEM;
//   * programmatic dependent launch: the weight loads, which depend on nothing
//     the previous kernel in the stream writes, start before
//     griddepcontrol.wait; reading x and writing out come after it, so
//     consecutive layers overlap one's tail with the next one's weight stream.
//   * x has a ring of its own (8 K tiles), apart from the weight ring: with
//     shared slots, quantising the second half of a CTA's K slice had to wait
//     for the MMAs of the first half, a round trip on every call's critical
//     path (dependency wait -> x -> MMAs -> reduction).
// Three shapes of the kernel: up to 16 tokens (8-stage weight ring, ~165 KB of
// shared memory), up to 64 tokens (6-stage weight ring) and up to 128 tokens
// (4-slot weight and activation rings, 512 TMEM columns), one CTA per SM.
// Warp roles: 0 = TMA producer (weights + weight scales), 1 = TMEM allocator
// and MMA issuer for the even K tiles, 10 = MMA issuer for the odd K tiles
// (each into its own accumulator; issuing a K tile's copies and MMAs takes one
// thread ~400 cycles, so two issuers halve that part of the call), 2..9 =
// activation quantiser, then (2..5) TMEM -> remote shared memory (the two
// accumulators summed in fixed order) and (2..9) the reduction.
// Every mbarrier wait is bounded; the cluster barrier is reached on every
// path, also after an expired wait.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mx_kernels.h"
#include "mx_layout.cuh"
#include "mx_ptx.cuh"
#include "mx_quant.cuh"

namespace mx {

namespace {

constexpr int kRows = 128;  // weight rows per CTA = MMA M
constexpr int kTK = 128;    // K elements per stage
constexpr int QTHREADS = 256;  // warps 2..9
constexpr int kMma2Warp = 2 + QTHREADS / 32;  // second MMA issuer (odd K tiles)
constexpr int THREADS = 64 + QTHREADS + 32;
constexpr int kWBytes = kRows * kTK;  // 16 KB

template <int MAXTOK_, int STAGES_, int XSTAGES_, int QB_, int MINB_>
struct DCfg {
  static constexpr int MAXTOK = MAXTOK_;
  static constexpr int STAGES = STAGES_;    // weight ring
  static constexpr int XSTAGES = XSTAGES_;  // activation ring (its own slots and barriers)
  static constexpr int QB = QB_;          // 32-element x blocks per quantiser thread per group
  static constexpr int MINB = MINB_;      // CTAs per SM the kernel is built for
  static constexpr int XBYTES = MAXTOK * kTK;
  static constexpr int OFF_W = 0;
  static constexpr int OFF_X = OFF_W + STAGES * kWBytes;
  static constexpr int OFF_SFW = OFF_X + XSTAGES * XBYTES;
  static constexpr int OFF_SFX = OFF_SFW + STAGES * kAtomBytes;
  static constexpr int OFF_RECV = OFF_SFX + XSTAGES * kAtomBytes;  // [S][n_mma][128/S] fp32
  static constexpr int RECV_BYTES = MAXTOK * kRows * 4;
  static constexpr int OFF_BAR = OFF_RECV + RECV_BYTES;
  // full_w, empty per weight stage; full_x, x_empty per activation slot; acc_full
  static constexpr int NUM_BARS = 2 * STAGES + 2 * XSTAGES + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
  static constexpr int T_ACC = 0;        // MAXTOK fp32 columns: even K tiles
  static constexpr int T_ACC1 = MAXTOK;  // odd K tiles
  static constexpr int T_SFW = 2 * MAXTOK;
  static constexpr int T_SFX = T_SFW + 4 * STAGES;
  static constexpr int T_END = T_SFX + 4 * STAGES;
  static constexpr int TMEM_COLS =
      T_END <= 32 ? 32 : (T_END <= 64 ? 64 : (T_END <= 128 ? 128 : (T_END <= 256 ? 256 : 512)));
  static_assert(T_END <= 512, "tensor memory");
  static_assert(MINB * SMEM_ALLOC <= 232448, "shared memory");
  static_assert(QTHREADS % kRows == 0, "each reduction thread owns one output column");
};

// Eight activation slots: at N = K = 4096 each CTA's K slice is 8 tiles at
// S = 4, so all of x is quantised in one pass right after the dependency wait
// instead of waiting for the MMAs of earlier tiles to free shared slots.  Up to
// 16 tokens the weight ring holds the whole 8-tile slice too (one CTA per SM):
// measured 8.45 us per call at M = 1 against 9.10 us for a 4-stage ring at two
// CTAs per SM, whose second half of the slice refilled on the critical path.
using SmallCfg = DCfg<16, 8, 8, 1, 1>;
// Up to 16 tokens where a CTA's K slice is longer than 8 tiles (no split at
// large N): an 11-stage weight ring, the most that fits beside the 8-slot
// activation ring (N = 14336, K = 4096: 14.2 -> 13.4 us at M = 1; at
// N = K = 4096 it measured 6.02 -> 6.12 us, so the 8-stage shape stays there).
using DeepCfg = DCfg<16, 11, 8, 1, 1>;
using LargeCfg = DCfg<64, 6, 8, 2, 1>;
// Up to 128 tokens (a prefill chunk): 4-slot rings of 16 KB weight tiles and
// 16 KB code tiles, a 64 KB receive buffer, two 128-column accumulators.
using WideCfg = DCfg<kDecodeMaxM, 4, 4, 2, 1>;

struct Args {
  const uint4* x;  // bf16 [M, K] as 16-byte chunks, or nullptr:
  const uint8_t* xq;  // pre-quantised E4M3 [M, K] and
  const uint8_t* xs;  // its scales [M, K/32], copied into the slots: row-major,
  int xs_packed;      // or (1) in the packed atom layout of mxfp8_quantize_packed
  const uint8_t* sfw;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  int M, N, K;
  int n_mma;   // MMA N: 16, 32 or 64 (>= M)
  int KT;      // K / 128
  int RTW;     // 128-row atom tiles of the weights
  int splits;  // cluster size S
  int wfmt;    // weight (A operand) element format
  uint8_t* yq;   // MXFP8 hand-off of the output (kHandOff): E4M3 [M, N] ...
  uint8_t* ysf;  // ... and its scales in packed atoms (one 128-row tile)
  int KTY;       // N / 128: K tiles of the hand-off's scale atoms
};

// kPreQ: x arrives pre-quantised (a.xq, a.xs) and is copied, not quantised;
// a separate instantiation, so that the bf16 path carries no branch for it
// (a run-time test cost that path ~0.25 us per call at N = K = 4096).
// kHandOff: the output is also quantised for the next layer (a.yq, a.ysf;
// a.out may then be null): needs N % 128 == 0, and the launcher splits K at
// most 4 ways, so that one warp holds the 32 columns of each block.
template <class C, bool kPreQ, bool kHandOff>
__global__ void __launch_bounds__(THREADS, C::MINB)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full_w = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full_w + C::STAGES;
  uint64_t* full_x = empty + C::STAGES;
  uint64_t* x_empty = full_x + C::XSTAGES;
  uint64_t* acc_full = x_empty + C::XSTAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int tile = blockIdx.x / a.splits;
  const int kt0 = static_cast<int>(static_cast<int64_t>(rank) * a.KT / a.splits);
  const int kt1 = static_cast<int>(static_cast<int64_t>(rank + 1) * a.KT / a.splits);
  const int nk = kt1 - kt0;  // >= 1 because splits <= KT

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_w[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::XSTAGES; ++s) {
      mbar_init(&full_x[s], QTHREADS / 32);  // one arrive per quantiser warp
      mbar_init(&x_empty[s], 1);
    }
    mbar_init(acc_full, 2);  // one commit per MMA issuer
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The bias of the output column this thread reduces (warps 2.. only): read
  // before the dependency wait, like the weights (the previous kernel in the
  // stream never writes it), so its latency is off the path after the MMAs
  // (measured: 6.27 -> 6.02 us per call at M = 1, 9.80 -> 9.48 at M = 64).
  float bias_n = 0.f;

  if (warp == 0) {
    // ------------------------------------------------ weight producer (TMA)
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int st = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&full_w[st], weight_tile_tx_bytes(kRows, a.wfmt) + kAtomBytes);
        tma_load_3d(smem + C::OFF_W + st * kWBytes, &tmW, &full_w[st], (kt0 + i) * kTK, tile * kRows, 0);
        bulk_load(smem + C::OFF_SFW + st * kAtomBytes,
                  a.sfw + (static_cast<int64_t>(kt0 + i) * a.RTW + tile) * kAtomBytes, kAtomBytes,
                  &full_w[st]);
        ++issued;
        if (i + 1 == min(nk, C::STAGES)) {
          launch_dependents();  // the next kernel may start loading
          // The rest of the slice waits for ring slots that the MMAs free only
          // after x is ready; ask L2 for it now.
          for (int j = C::STAGES; j < nk; ++j) {
            prefetch_tile_l2(&tmW, (kt0 + j) * kTK, tile * kRows, 0);
            prefetch_bulk_l2(a.sfw + (static_cast<int64_t>(kt0 + j) * a.RTW + tile) * kAtomBytes, kAtomBytes);
          }
        }
      }
      if (*abort_flag) {
        for (int s = 0; s < C::STAGES && s < issued; ++s) {
          const int last = ((issued - 1 - s) / C::STAGES) * C::STAGES + s;
          mbar_wait(&full_w[s], static_cast<uint32_t>((last / C::STAGES) & 1), nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMma2Warp) {
    // ------------------------------------------------ MMA issuers: even K tiles
    // into one accumulator, odd into another (summed in fixed order below)
    if (lane == 0) {
      const int par = warp == 1 ? 0 : 1;
      const uint32_t t_acc = tmem + (par ? C::T_ACC1 : C::T_ACC);
      const uint32_t idesc0 = idesc_with_types(idesc_mxf8(kRows, a.n_mma), a.wfmt, kFmtE4M3);
      bool ok = true;
      for (int i = par; i < nk && ok; i += 2) {
        const int st = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        const int xs = i % C::XSTAGES;
        const uint32_t xph = (i / C::XSTAGES) & 1;
        if (!mbar_wait(&full_w[st], ph, abort_flag) || !mbar_wait(&full_x[xs], xph, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // TMEM scale slots follow the weight stage: the copies run on the
        // tensor pipe in order behind the MMAs that read the slot before.
        const uint32_t t_sfw = tmem + C::T_SFW + st * 4;
        const uint32_t t_sfx = tmem + C::T_SFX + st * 4;
        tc_cp_sf(t_sfw, sdesc_sf(smem_u32(smem + C::OFF_SFW + st * kAtomBytes)));
        tc_cp_sf(t_sfx, sdesc_sf(smem_u32(smem + C::OFF_SFX + xs * kAtomBytes)));
        const uint64_t ad = sdesc_kmajor_sw128(smem_u32(smem + C::OFF_W + st * kWBytes));
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(smem + C::OFF_X + xs * C::XBYTES));
#pragma unroll
        for (int kk = 0; kk < kTK / 32; ++kk)
          tc_mma_mxf8(t_acc, ad + 2 * kk, bd + 2 * kk, idesc_with_sf_id(idesc0, kk, kk), t_sfw, t_sfx,
                      i >= 2 || kk != 0);
        tc_commit(&empty[st]);
        tc_commit(&x_empty[xs]);
      }
      if (ok) tc_commit(acc_full);
      else __nanosleep(200000);  // let issued tensor-core work retire
    }
    __syncwarp();
  } else if (warp < kMma2Warp) {
    // Token rows M .. n_mma - 1 are zero in every K tile: write their codes and
    // scale bytes once, before the dependency wait, and quantise only rows < M
    // afterwards (a zero block quantises to byte 0 and zero codes, so this is
    // what quantising them would write).  Rows < M are never touched here.
    {
      const int tz = threadIdx.x - 64;
      const int zrows = a.n_mma - a.M;
      for (int idx = tz; idx < C::XSTAGES * zrows * 8; idx += QTHREADS) {
        const int xs = idx / (zrows * 8);
        const int rem = idx - xs * zrows * 8;
        const int row = a.M + rem / 8;
        *reinterpret_cast<uint4*>(smem + C::OFF_X + xs * C::XBYTES + row * 128 + (rem & 7) * 16) =
            make_uint4(0, 0, 0, 0);
        if ((rem & 7) == 0)
          *reinterpret_cast<uint32_t*>(smem + C::OFF_SFX + xs * kAtomBytes + (row & 31) * 16 + (row >> 5) * 4) = 0u;
      }
    }
    {
      // the column this thread adds the bias to: in the reduction below, or
      // (one CTA per tile) in the epilogue's direct store, warps 2..5
      const int per = kRows / a.splits;
      const int n = a.splits == 1 ? tile * kRows + (warp & 3) * 32 + lane
                                  : tile * kRows + static_cast<int>(rank) * per + (threadIdx.x - 64) % per;
      if (a.bias != nullptr && n < a.N) bias_n = __bfloat162float(a.bias[n]);
    }
    // x is written by the previous kernel in the stream: wait for it to finish.
    grid_dependency_wait();
    // ------------------------------------------------ activation quantiser
    // A task is one 32-element block of x: K tile i, token row r < M, block j
    // of the tile's four, one lane per block (quantize_block32, as in the
    // standalone quantize kernel; a lane per quarter block with shuffles took
    // ~7 us for 64 tokens).  One group = G K tiles = G * M * 4 tasks, at most
    // QB per thread.  Rows M .. n_mma - 1 were zeroed above.
    const int t = threadIdx.x - 64;
    const int per_tile = a.M * 4;
    // A group's slots must all be free at once while the MMA still owns the
    // others, so a group spans at most half the activation ring.
    const int G = max(1, min(C::XSTAGES / 2, (QTHREADS * C::QB) / per_tile));
    const int per_group = G * per_tile;  // <= QTHREADS * QB
    auto load_group = [&](int g, uint4 (&dst)[C::QB][4]) {
#pragma unroll
      for (int u = 0; u < C::QB; ++u) {
        const int task = t + u * QTHREADS;
        const int ti = task / per_tile;
        const int i = g * G + ti;
        const int rem = task - ti * per_tile;
        const bool valid = task < per_group && i < nk;
        const int64_t e0 = static_cast<int64_t>(rem >> 2) * a.K + (kt0 + i) * kTK + (rem & 3) * 32;
        if (kPreQ) {
          // pre-quantised: the block's 32 codes and its scale byte
          const uint4* src = reinterpret_cast<const uint4*>(a.xq + e0);
          dst[u][0] = valid ? __ldg(src) : make_uint4(0, 0, 0, 0);
          dst[u][1] = valid ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
          const int64_t so = a.xs_packed ? sf_packed_offset(0, rem >> 2, (kt0 + i) * 4 + (rem & 3),
                                                            (a.M + kAtomRows - 1) / kAtomRows, a.KT)
                                         : e0 / 32;
          dst[u][2].x = valid ? static_cast<uint32_t>(__ldg(a.xs + so)) : 0u;
        } else {
          const uint4* src = a.x + e0 / 8;
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[u][k] = valid ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
        }
      }
    };
    // Wait for the group's ring slots, quantise it into them, signal the MMA.
    auto quantize_group = [&](int g, const uint4 (&cur)[C::QB][4]) -> bool {
      for (int i = g * G; i < min(nk, (g + 1) * G); ++i)
        if (!mbar_wait(&x_empty[i % C::XSTAGES], ((i / C::XSTAGES) & 1) ^ 1u, abort_flag)) return false;
#pragma unroll
      for (int u = 0; u < C::QB; ++u) {
        const int task = t + u * QTHREADS;
        const int ti = task / per_tile;
        const int i = g * G + ti;
        if (task >= per_group || i >= nk) break;
        const int rem = task - ti * per_tile;
        const int row = rem >> 2, j = rem & 3;
        uint4 c0, c1;
        uint32_t sbyte;
        if (kPreQ) {
          c0 = cur[u][0];
          c1 = cur[u][1];
          sbyte = cur[u][2].x;
        } else {
          sbyte = quantize_block32(cur[u], c0, c1);
        }
        const int xs = i % C::XSTAGES;
        uint8_t* xrow = smem + C::OFF_X + xs * C::XBYTES + row * 128;
        // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8);
        // block j is chunks 2j and 2j + 1 of its row
        *reinterpret_cast<uint4*>(xrow + (((2 * j) ^ (row & 7)) << 4)) = c0;
        *reinterpret_cast<uint4*>(xrow + (((2 * j + 1) ^ (row & 7)) << 4)) = c1;
        smem[C::OFF_SFX + xs * kAtomBytes + (row & 31) * 16 + (row >> 5) * 4 + j] = static_cast<uint8_t>(sbyte);
      }
      fence_proxy_async_smem();
      // One arrive per warp: arrivals on a barrier are serialised.
      __syncwarp();
      if ((threadIdx.x & 31) == 0)
        for (int i = g * G; i < min(nk, (g + 1) * G); ++i) mbar_arrive(&full_x[i % C::XSTAGES]);
      return true;
    };
    const int ngroups = (nk + G - 1) / G;
    uint4 buf0[C::QB][4], buf1[C::QB][4];  // two register sets: load one group ahead
    load_group(0, buf0);
    for (int g = 0; g < ngroups; g += 2) {
      if (g + 1 < ngroups) load_group(g + 1, buf1);
      if (!quantize_group(g, buf0)) break;
      if (g + 1 >= ngroups) break;
      if (g + 2 < ngroups) load_group(g + 2, buf0);
      if (!quantize_group(g + 1, buf1)) break;
    }

    // ------------------------------------------------ epilogue, one CTA per tile: TMEM -> out
    // (the same sum, in the same order, as the reduction below with S = 1;
    // measured 14.8 -> 14.1 us per call at M = 1, N = 14336)
    if (a.splits == 1 && warp < 6 && mbar_wait(acc_full, 0, abort_flag)) {
      tc_fence_after();
      const int quad = warp & 3;
      const int n = tile * kRows + quad * 32 + lane;
      const uint32_t lrow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      for (int c = 0; c < a.n_mma; c += 16) {
        uint32_t r[16], r1[16];
        tmem_ld_32x32b_x16(lrow + C::T_ACC + c, r);
        tmem_ld_32x32b_x16(lrow + C::T_ACC1 + c, r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float v = nk > 1 ? __uint_as_float(r[j]) + __uint_as_float(r1[j]) : __uint_as_float(r[j]);
          if constexpr (kHandOff) {
            if (c + j < a.M) {  // the same row in every lane: the warp is one block
              const __nv_bfloat16 yb = __float2bfloat16_rn((0.f + v) + bias_n);
              if (a.out != nullptr) a.out[static_cast<int64_t>(c + j) * a.N + n] = yb;
              uint32_t sb;
              const uint32_t code = quantize_lane_block(__bfloat16_as_ushort(yb), &sb);
              a.yq[static_cast<int64_t>(c + j) * a.N + n] = static_cast<uint8_t>(code);
              if (lane == 0) a.ysf[sf_packed_offset(0, c + j, n >> 5, 1, a.KTY)] = static_cast<uint8_t>(sb);
            }
          } else {
            if (c + j < a.M && n < a.N)
              a.out[static_cast<int64_t>(c + j) * a.N + n] = __float2bfloat16_rn((0.f + v) + bias_n);
          }
        }
      }
    }
    // ------------------------------------------------ epilogue, K split: TMEM -> owner's receive buffer
    if (a.splits > 1 && warp < 6 && mbar_wait(acc_full, 0, abort_flag)) {
      tc_fence_after();
      const int quad = warp & 3;
      const int wrow = quad * 32 + lane;  // weight row within the tile = TMEM lane
      const int per = kRows / a.splits;
      const uint32_t owner = static_cast<uint32_t>(wrow / per);
      const int nl = wrow - static_cast<int>(owner) * per;
      const uint32_t dst = map_shared_rank(smem_u32(smem + C::OFF_RECV), owner) +
                           static_cast<uint32_t>(((rank * a.n_mma) * per + nl) * 4);
      for (int c = 0; c < a.n_mma; c += 16) {
        uint32_t r[16], r1[16];
        const uint32_t lrow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        tmem_ld_32x32b_x16(lrow + C::T_ACC + c, r);
        tmem_ld_32x32b_x16(lrow + C::T_ACC1 + c, r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float v = nk > 1 ? __uint_as_float(r[j]) + __uint_as_float(r1[j]) : __uint_as_float(r[j]);
          st_shared_cluster_u32(dst + static_cast<uint32_t>((c + j) * per * 4), __float_as_uint(v));
        }
      }
    }
  }

  // ------------------------------------------------ split-K reduction (owner sums)
  tc_fence_before();
  cluster_sync();  // all partials have landed in their owners' receive buffers
  if (a.splits > 1 && threadIdx.x >= 64 && threadIdx.x < 64 + QTHREADS && !*abort_flag) {
    const int t = threadIdx.x - 64;
    const int per = kRows / a.splits;
    const float* recv = reinterpret_cast<const float*>(smem + C::OFF_RECV);
    // QTHREADS is a multiple of per, so each thread keeps one output column n
    const int nl = t % per;
    const int n = tile * kRows + static_cast<int>(rank) * per + nl;
    const float bias = bias_n;  // loaded before the dependency wait (same n)
    if (n < a.N) {
#pragma unroll 4
      for (int m = t / per; m < a.M; m += QTHREADS / per) {
        float acc = 0.f;
        for (int s2 = 0; s2 < a.splits; ++s2) acc += recv[(s2 * a.n_mma + m) * per + nl];
        if constexpr (kHandOff) {
          // per >= 32: the warp holds one 32-column block of row m
          const __nv_bfloat16 yb = __float2bfloat16_rn(acc + bias);
          if (a.out != nullptr) a.out[static_cast<int64_t>(m) * a.N + n] = yb;
          uint32_t sb;
          const uint32_t code = quantize_lane_block(__bfloat16_as_ushort(yb), &sb);
          a.yq[static_cast<int64_t>(m) * a.N + n] = static_cast<uint8_t>(code);
          if (lane == 0) a.ysf[sf_packed_offset(0, m, n >> 5, 1, a.KTY)] = static_cast<uint8_t>(sb);
        } else {
          a.out[static_cast<int64_t>(m) * a.N + n] = __float2bfloat16_rn(acc + bias);
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

template <class C>
cudaError_t prepare_cfg(const char** msg) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    void (*const kernels[4])(const CUtensorMap, const Args) = {
        gemm_decode_kernel<C, false, false>, gemm_decode_kernel<C, true, false>, gemm_decode_kernel<C, false, true>,
        gemm_decode_kernel<C, true, true>};
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
      e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) {
      *msg = "cudaFuncSetAttribute(max dynamic shared memory) failed";
      return e;
    }
    attr_set[dev] = true;
  }
  return cudaSuccess;
}

// Clusters of `splits` CTAs of this kernel that fit on the GPU at once (asked
// of the driver once per device and cluster size).
template <class C>
int max_active_clusters(int splits) {
  static int cache[64][4] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int slot = splits == 8 ? 3 : (splits == 4 ? 2 : (splits == 2 ? 1 : 0));
  if (dev < 0 || dev >= 64) return 0;
  if (cache[dev][slot] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(splits), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_decode_kernel<C, false, false>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();  // clear the sticky-free error state of the failed query
      n = -1;
    }
    cache[dev][slot] = n;
  }
  return cache[dev][slot];
}

template <class C, bool kPreQ, bool kHandOff>
cudaError_t launch_cfg(const CUtensorMap& mw, const Args& a, int grid, cudaStream_t stream,
                       const char** msg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_decode_kernel<C, kPreQ, kHandOff>, mw, a);
  if (e != cudaSuccess) *msg = "decode GEMM launch failed";
  return e;
}

}  // namespace

namespace {

// The largest K split (at most 8, at most one per K tile) whose clusters all
// fit on the GPU at once, so that every CTA streams its weights from the start.
template <class C>
int k_splits(int tiles, int KT, int sms) {
  int splits = 8;
  while (splits > 1) {
    const int fit = max_active_clusters<C>(splits);
    const bool fits = fit > 0 ? tiles <= fit : tiles * splits <= C::MINB * sms;
    if (splits <= KT && fits) break;
    splits >>= 1;
  }
  return splits;
}

}  // namespace

int decode_k_splits(int64_t M, int64_t N, int64_t K, int sms) {
  const char* msg = "";
  const int tiles = static_cast<int>(ceil_div(N, kRows));
  const int KT = static_cast<int>(K / kTK);
  if (M <= SmallCfg::MAXTOK)
    return prepare_cfg<SmallCfg>(&msg) == cudaSuccess ? k_splits<SmallCfg>(tiles, KT, sms) : 1;
  if (M <= LargeCfg::MAXTOK)
    return prepare_cfg<LargeCfg>(&msg) == cudaSuccess ? k_splits<LargeCfg>(tiles, KT, sms) : 1;
  return prepare_cfg<WideCfg>(&msg) == cudaSuccess ? k_splits<WideCfg>(tiles, KT, sms) : 1;
}

namespace {

template <class C>
cudaError_t launch_with(const CUtensorMap& mw, Args& a, bool preq, int sms, cudaStream_t stream,
                        const char** msg) {
  cudaError_t e = prepare_cfg<C>(msg);
  if (e != cudaSuccess) return e;
  a.splits = k_splits<C>(a.RTW, a.KT, sms);
  if (a.yq != nullptr) {
    // the hand-off needs whole 32-column blocks in one owner: at most 4 ways
    if (a.N % 128 != 0) {
      *msg = "small-M hand-off: needs N % 128 == 0";
      return cudaErrorInvalidValue;
    }
    if (a.splits > 4) a.splits = 4;
    return preq ? launch_cfg<C, true, true>(mw, a, a.RTW * a.splits, stream, msg)
                : launch_cfg<C, false, true>(mw, a, a.RTW * a.splits, stream, msg);
  }
  const int grid = a.RTW * a.splits;
  return preq ? launch_cfg<C, true, false>(mw, a, grid, stream, msg)
              : launch_cfg<C, false, false>(mw, a, grid, stream, msg);
}

}  // namespace

cudaError_t launch_gemm_decode(const DecodeProblem& p, int sms, cudaStream_t stream, const char** msg) {
  CUtensorMap mw;
  cudaError_t e = make_operand_map(&mw, p.w, 1, p.N, p.K, kRows, msg, p.wfmt);
  if (e != cudaSuccess) return e;

  Args a;
  a.x = static_cast<const uint4*>(p.x);
  a.xq = p.xq;
  a.xs = p.xs;
  a.xs_packed = p.xs_packed;
  a.yq = p.yq;
  a.ysf = p.ysf;
  a.KTY = static_cast<int>(p.N / 128);
  a.sfw = p.sfw;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.M = static_cast<int>(p.M);
  a.N = static_cast<int>(p.N);
  a.K = static_cast<int>(p.K);
  a.wfmt = p.wfmt;
  // MMA N: a power of two (shifts in the quantiser), at least M
  a.n_mma = p.M <= 16 ? 16 : (p.M <= 32 ? 32 : (p.M <= 64 ? 64 : 128));
  a.KT = static_cast<int>(p.K / kTK);
  a.RTW = static_cast<int>(ceil_div(p.N, kAtomRows));
  const bool preq = p.xq != nullptr;
  if (a.n_mma <= SmallCfg::MAXTOK) {
    // the same split either way (one CTA per SM, the same cluster sizes)
    e = prepare_cfg<SmallCfg>(msg);
    if (e != cudaSuccess) return e;
    if (a.KT / k_splits<SmallCfg>(a.RTW, a.KT, sms) > SmallCfg::STAGES)
      return launch_with<DeepCfg>(mw, a, preq, sms, stream, msg);
    return launch_with<SmallCfg>(mw, a, preq, sms, stream, msg);
  }
  if (a.n_mma <= LargeCfg::MAXTOK) return launch_with<LargeCfg>(mw, a, preq, sms, stream, msg);
  return launch_with<WideCfg>(mw, a, preq, sms, stream, msg);
}

cudaError_t take_status_decode(unsigned int* out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace mx
