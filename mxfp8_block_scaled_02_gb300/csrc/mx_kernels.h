// mx_kernels.h - host-side launchers shared between the translation units of
// libmxfp8.so.  Internal: not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mx {

// quantize.cu.  The kernels index 32-element blocks and 4-byte scale words
// with 32-bit integers: the host refuses larger problems before launching.
constexpr int64_t kMaxBlocks32 = 0x7FFFFFFFll;
// early_trigger: let the next kernel in the stream start before this one ends
// (programmatic dependent launch).  Only for the activation quantise / scale
// repack inside the linear layer: the GEMM that follows reads their output
// after its dependency wait.  Never for weights (the GEMMs load weights and
// weight scales before that wait).
cudaError_t launch_quantize(const void* x, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                            bool packed_scales, int64_t B, int64_t rows_per_b, int sms,
                            cudaStream_t stream, bool early_trigger);
cudaError_t launch_sf_pack(const uint8_t* src, int64_t B, int64_t R, int64_t K, uint8_t* dst,
                           int sms, cudaStream_t stream, bool early_trigger);
// MXFP6 weights: bf16 -> one FP6 (or E4M3) code per byte + row-major scales
// (fmt: kFmtE4M3 / kFmtE2M3 / kFmtE3M2 of mx_quant.cuh), and the repack of n
// FP6 codes (n % 16 == 0) into the packed 6-bit layout (3n/4 bytes).
cudaError_t launch_quantize_weights(const void* x, int64_t rows, int64_t K, int fmt, uint8_t* q, uint8_t* s,
                                    int sms, cudaStream_t stream);
cudaError_t launch_fp6_pack(const uint8_t* codes, int64_t n, uint8_t* out, int sms, cudaStream_t stream);
cudaError_t launch_sf_unpack(const uint8_t* src, int64_t B, int64_t R, int64_t K, uint8_t* dst,
                             int sms, cudaStream_t stream);
cudaError_t take_status_quantize(unsigned int* out);

// gemm.cu: the large-M path.  A = activations [B, M, K] E4M3, Bw = weights
// [B, N, K] E4M3, both K-major; sfa / sfb are packed scale atoms.
struct GemmProblem {
  const uint8_t* a;
  const uint8_t* w;
  const uint8_t* sfa;
  const uint8_t* sfb;
  const void* bias;  // bf16 [N] or nullptr
  void* out;         // bf16 [B, M, N]
  int64_t B, M, N, K;
  int tiles = 0;     // 0: by M (CTA pairs when M > 128); 1: one CTA per 128 x 256 tile; 2: CTA pairs
  // MXFP8 hand-off (mx_epilogue.cuh): when yq is set the epilogue also writes
  // the output quantised, codes [B, M, N] to yq and packed scale atoms of
  // (B, M, N) to ysf (N % 128 == 0); out may then be nullptr (no bf16 output).
  uint8_t* yq = nullptr;
  uint8_t* ysf = nullptr;
  int wfmt = 0;      // weight element format: 0 E4M3, 1 E2M3, 2 E3M2 (packed 6-bit, see make_operand_map)
  // split-K (CTA-pair kernel only): with part set and splits > 1, each tile's K
  // range is split over `splits` pairs, the fp32 partials go to part
  // ([splits * B][M][N]) and a reduce kernel writes out / the hand-off.
  float* part = nullptr;
  int splits = 1;
  // 1: sfa is the caller's row-major activation scales [B, M, K/32] instead of
  // packed atoms (CTA-pair kernel only: its scale writers gather the atom lines)
  int sfa_rowmajor = 0;
};
// Whether launch_gemm_prefill runs p on the CTA-pair kernel (else one CTA per
// 128 x 256 tile).
bool gemm_prefill_uses_pair(const GemmProblem& p, int sms);
// K splits the linear layer uses for a shape (1 = none): enough to give about
// 64 CTA pairs work when there are at most 16 tiles of 256 x 256, with at least
// four 128-wide K tiles per split and at most 8 splits.  A function of the
// shape alone, so the workspace size is known before the call.
int splitk_splits(int64_t B, int64_t M, int64_t N, int64_t K);
// out[b, m, n] = bf16(sum over s of part[s][b][m][n] in order s = 0.. + bias[n]),
// and / or the MXFP8 hand-off of those bf16 values (splitk.cu).
cudaError_t launch_splitk_reduce(const float* part, int splits, int64_t B, int64_t M, int64_t N, const void* bias,
                                 void* out, uint8_t* yq, uint8_t* ysf, int sms, cudaStream_t stream);
// fp32 [Z][M][N] split-K partials, box {16 columns, 32 rows, 1} (gemm.cu).
cudaError_t make_partial_map(CUtensorMap* map, float* part, int64_t Z, int64_t M, int64_t N, const char** msg);
// Returns cudaSuccess, or the failing CUDA error; *msg names the failing step.
cudaError_t launch_gemm_prefill(const GemmProblem& p, int sms, cudaStream_t stream, const char** msg);
cudaError_t take_status_gemm(unsigned int* out);
// gemm_pair.cu: 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2).
cudaError_t launch_gemm_pair(const GemmProblem& p, int sms, cudaStream_t stream, const char** msg);
cudaError_t take_status_pair(unsigned int* out);
// bf16 [B][M][N] output map, box {32 columns, 32 rows, 1} (gemm.cu).
cudaError_t make_output_map(CUtensorMap* map, void* out, int64_t B, int64_t M, int64_t N, const char** msg);
// 3-D TMA map over [B][rows][K] E4M3 bytes, box {128, box_rows, 1}, 128-byte
// swizzle.  fmt != 0: the operand is packed 6-bit FP6 codes (3K/4 bytes per
// row, CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B), which the copy expands to 16
// bytes per 16 codes in shared memory: the same tile shape as E4M3.
cudaError_t make_operand_map(CUtensorMap* map, const uint8_t* base, int64_t B, int64_t rows,
                             int64_t K, int box_rows, const char** msg, int fmt = 0);

// gemm_fq.cu: the linear layer with x quantised inside the GEMM (bf16 x
// [B, M, K] read once, no quantised copy in memory), one CTA per 128 x 256
// output tile: for shapes whose fused_quantize_tiles(B, M, N) fit on the GPU
// at once (<= the SM count), N % 8 == 0, K % 128 == 0.
struct FusedProblem {
  const void* x;      // bf16 [B, M, K]
  const uint8_t* w;   // weights [B, N, K] (E4M3, or packed FP6 by wfmt)
  const uint8_t* sfw; // packed weight scale atoms
  const void* bias;   // bf16 [N] or nullptr
  void* out;          // bf16 [B, M, N]
  int64_t B, M, N, K;
  int wfmt = 0;
};
int64_t fused_quantize_tiles(int64_t B, int64_t M, int64_t N);
cudaError_t launch_gemm_fq(const FusedProblem& p, int sms, cudaStream_t stream, const char** msg);
cudaError_t take_status_fq(unsigned int* out);

// gemm_decode.cu: the small-M path (M <= 64, B = 1, bf16 x): weights on the
// MMA's M side, activations quantised inside the kernel, split-K across a
// thread-block cluster with a fixed-order reduction in distributed shared memory.
struct DecodeProblem {
  const void* x;     // bf16 [M, K], or nullptr when xq / xs are given
  const uint8_t* w;  // E4M3 [N, K]
  const uint8_t* sfw;
  const void* bias;  // bf16 [N] or nullptr
  void* out;         // bf16 [M, N]
  int64_t M, N, K;
  int wfmt = 0;      // weight element format, as GemmProblem::wfmt
  const uint8_t* xq = nullptr;  // pre-quantised x: E4M3 [M, K] ...
  const uint8_t* xs = nullptr;  // ... and its E8M0 scales [M, K/32]: row-major,
  int xs_packed = 0;            // or (1) packed atoms as mxfp8_quantize_packed writes them
  uint8_t* yq = nullptr;        // MXFP8 hand-off of the output (E4M3 [M, N]) and its
  uint8_t* ysf = nullptr;       // packed scales; out may then be null (N % 128 == 0, K split <= 4)
};
constexpr int kDecodeMaxM = 128;  // largest M the small-M kernel takes
// The K split (cluster size) launch_gemm_decode uses for this shape; 1 = none.
int decode_k_splits(int64_t M, int64_t N, int64_t K, int sms);
cudaError_t launch_gemm_decode(const DecodeProblem& p, int sms, cudaStream_t stream, const char** msg);
cudaError_t take_status_decode(unsigned int* out);

// debug.cu
cudaError_t launch_expire_wait(uint64_t timeout_ns, cudaStream_t stream);
cudaError_t take_status_debug(unsigned int* out);

// api.cu: record the text mxfp8_last_error() returns on this thread.
void set_last_error(const char* msg);

// Driver entry point for cuTensorMapEncodeTiled (resolved once, via the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

}  // namespace mx
