/*
 * mxfp8.h - C ABI of libmxfp8.so, the GB300 (sm_103a) W8A8 MXFP8 linear layer.
 *
 * The layer (sources are vLLM API pages, cited by page and section):
 *   - "CompressedTensorsW8A8Mxfp8" (compressed_tensors_w8a8_mxfp8 page), class
 *     docstring "MXFP8 format": FP8 E4M3 elements, one uint8 E8M0 scale per
 *     32 consecutive elements along K, activations quantised at run time;
 *     create_weights: weight [N, K] E4M3, weight_scale [N, K/32] uint8.
 *   - "AiterFlyDSLMxfp8LinearKernel" (aiter_flydsl page), class docstring and
 *     apply_weights: activation scales row-major [M, K/32]; the activation is
 *     either quantised inside the layer or handed over pre-quantised; output
 *     in the input dtype (bf16), then "+ bias".
 *   - "Mxfp8LinearLayerConfig" (Mxfp8LinearKernel page): weight_shape (N, K)
 *     and bmm_batch_size (a batched layer).
 *   - "Mxfp8LinearKernel.process_weights_after_loading" (Mxfp8LinearKernel
 *     page): a one-time rewrite of the weights after loading.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device (or managed) pointers on the
 *     current device; the caller allocates and frees every buffer, including
 *     the workspace.  The library allocates no memory and keeps no per-layer
 *     state.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and returns without synchronising.  Nothing throws across the ABI.
 *   - Argument problems are found before any launch and return
 *     MXFP8_ERR_INVALID_ARG or MXFP8_ERR_UNSUPPORTED; a device that is not
 *     sm_103 returns MXFP8_ERR_ARCH; a failed CUDA call returns MXFP8_ERR_CUDA.
 *     mxfp8_last_error() then describes the problem (thread-local text).
 *   - Every wait inside a kernel is bounded in time.  A wait that runs out sets
 *     a device status word and the kernel returns; mxfp8_check() reports it as
 *     MXFP8_ERR_TIMEOUT.
 *   - Sizes are element counts.  Tensors are row-major and dense.
 *   - E4M3 codes and E8M0 scales are passed as bytes (uint8_t).  bf16 values are
 *     passed as raw 16-bit patterns (const void*).
 */
#ifndef MXFP8_H
#define MXFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* mxfp8_stream_t;

typedef enum {
  MXFP8_OK = 0,
  MXFP8_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer      */
  MXFP8_ERR_UNSUPPORTED = 2, /* valid request this library does not implement */
  MXFP8_ERR_ARCH = 3,        /* current device is not sm_103                   */
  MXFP8_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed           */
  MXFP8_ERR_TIMEOUT = 5      /* a bounded in-kernel wait ran out               */
} mxfp8_status;

#define MXFP8_BLOCK_SIZE 32

/* Text for the last non-OK status returned on this thread ("" if none). */
const char* mxfp8_last_error(void);

/* ABI version, currently 1. */
int mxfp8_version(void);

/*
 * mxfp8_quantize - dynamic MXFP8 quantisation of bf16 rows.
 *   Source: "AiterFlyDSLMxfp8LinearKernel.apply_weights" (aiter_flydsl page),
 *   the mxfp8_e4m3_quantize step and its scale-shape assert; arithmetic per the
 *   OCP MX v1.0 rule (section 6.3): per 32-block, e = floor(log2 amax) - 8
 *   clamped to [-127, 127], scale byte = e + 127, element = E4M3(x / 2^e) with
 *   round-to-nearest-even and saturation to +-448.  An all-zero block gets
 *   scale byte 0; a block holding Inf or NaN gets 0xFF and elements 0x7F.
 *   x_bf16  : device, [rows, K] bf16, 16-byte aligned.
 *   x_q     : device, [rows, K] E4M3 codes out, 16-byte aligned.
 *   x_scale : device, [rows, K/32] E8M0 bytes out (row-major), 16-byte aligned.
 *   rows >= 0 (0 is a no-op), K > 0 and K % 32 == 0; rows * K/32 above
 *   2^31 - 1 blocks returns MXFP8_ERR_UNSUPPORTED (split the call).
 */
mxfp8_status mxfp8_quantize(const void* x_bf16, int64_t rows, int64_t K, uint8_t* x_q,
                            uint8_t* x_scale, mxfp8_stream_t stream);

/*
 * mxfp8_packed_sizes - bytes of the packed weight blobs written by
 * mxfp8_process_weights for B batches of an [N, K] layer (B = 1 when not
 * batched).  The sizes depend only on (B, N, K), so callers may persist and
 * reload the blobs as plain bytes.
 */
mxfp8_status mxfp8_packed_sizes(int64_t B, int64_t N, int64_t K, size_t* w_bytes,
                                size_t* sf_bytes);

/*
 * mxfp8_process_weights - one-time repack of loaded MXFP8 weights.
 *   Source: "Mxfp8LinearKernel.process_weights_after_loading" (Mxfp8LinearKernel
 *   page) and "CompressedTensorsW8A8Mxfp8.create_weights" (weight [N, K] E4M3,
 *   weight_scale [N, K/32] uint8).
 *   w        : device, [B, N, K] E4M3 codes (row-major, K contiguous).
 *   w_scale  : device, [B, N, K/32] E8M0 bytes (row-major), exactly K/32
 *              per row (a checkpoint whose scales are padded is sliced to
 *              [:N, :K/32] and made contiguous by the caller first).
 *   w_packed : device, w_bytes out: the E4M3 codes, K-major as the tensor cores
 *              read them (the same bytes as w; w_packed == w is allowed).
 *   sf_packed: device, sf_bytes out: the scales in 512-byte atoms of 128 rows x
 *              4 blocks, the tensor cores' scale-factor layout; padding is zero.
 *   B >= 1, N > 0, K > 0, K % 32 == 0.  Every pointer 16-byte aligned
 *   (MXFP8_ERR_INVALID_ARG otherwise, before any launch).  More than 2^31 - 1
 *   scale blocks returns MXFP8_ERR_UNSUPPORTED.
 */
mxfp8_status mxfp8_process_weights(const uint8_t* w, const uint8_t* w_scale, int64_t B,
                                   int64_t N, int64_t K, uint8_t* w_packed,
                                   uint8_t* sf_packed, mxfp8_stream_t stream);

/*
 * mxfp8_unpack_scales - exact inverse of the scale part of
 * mxfp8_process_weights: sf_packed -> row-major [B, N, K/32].  Used to check
 * the repack bit for bit (like row_major_weight on the aiter_flydsl page, which
 * inverts that backend's weight shuffle).
 */
mxfp8_status mxfp8_unpack_scales(const uint8_t* sf_packed, int64_t B, int64_t N, int64_t K,
                                 uint8_t* w_scale, mxfp8_stream_t stream);

/*
 * mxfp8_workspace_size - device workspace bytes mxfp8_linear needs for this
 * problem (the quantised activations and their packed scales, plus the
 * split-K partials, 4 * splits * B * M * N bytes, when the shape is split).
 * x_is_quantized = 1 when the caller passes x_q/x_scale.
 */
mxfp8_status mxfp8_workspace_size(int64_t B, int64_t M, int64_t N, int64_t K,
                                  int x_is_quantized, size_t* bytes);

/*
 * mxfp8_linear - out[b, m, n] = bf16( sum_k deq(x)[b, m, k] * deq(w)[b, n, k]
 *                                     + bias[n] ).
 *   Source: "AiterFlyDSLMxfp8LinearKernel.apply_weights" (aiter_flydsl page):
 *   quantise x (or take the pre-quantised QuantizedActivation data/scale),
 *   block-scaled GEMM against the processed weight, output in the input dtype,
 *   then + bias; "Mxfp8LinearLayerConfig.bmm_batch_size" for B > 1 (B
 *   independent products, one shared bias).
 *   Exactly one input form:
 *     x_bf16            : device, [B, M, K] bf16 (quantised inside the call), or
 *     x_q and x_scale   : device, [B, M, K] E4M3 and [B, M, K/32] E8M0 row-major.
 *   w_packed, sf_packed : device, from mxfp8_process_weights with the same B, N, K.
 *   bias_bf16           : device, [N] bf16, or NULL for no bias.
 *   out_bf16            : device, [B, M, N] bf16 out.
 *   workspace           : device, >= mxfp8_workspace_size() bytes (may be NULL
 *                         when that size is 0); 256-byte aligned.
 *   The accumulation is fp32 on the tensor cores and the result is rounded once
 *   to bf16 after the bias add.  Requirements: B >= 1, M >= 0 (0 is a no-op),
 *   N > 0 with N % 8 == 0, K > 0 with K % 128 == 0 (else MXFP8_ERR_UNSUPPORTED),
 *   all pointers (x_scale included) 16-byte aligned (else
 *   MXFP8_ERR_INVALID_ARG), at most 2^31 - 1 scale blocks in x and in w.
 *   Stream ordering: the GEMM kernels are launched with programmatic stream
 *   serialization.  When the kernel before them in the stream triggers its
 *   dependents early (griddepcontrol.launch_dependents), they may read
 *   w_packed, sf_packed and bias before that kernel ends; x, x_q, x_scale
 *   and out are touched only after it has finished.  The quantise step inside
 *   a linear call is launched the same way and touches nothing before the
 *   kernel ahead of it has finished.  Of this library's
 *   kernels, only these trigger early: the quantise / activation-scale repack
 *   step inside mxfp8_linear, mxfp8_linear_path and mxfp8_linear_noalloc
 *   (whose output only the same call's GEMM reads, after its wait), the
 *   CTA-pair GEMM when it splits K (whose partials only the same call's
 *   reduce reads, after its wait), and the small-M GEMM (whose output the
 *   next layer reads as x, after its wait).
 *   The standalone calls (mxfp8_quantize, mxfp8_quantize_packed,
 *   mxfp8_pack_scales, mxfp8_process_weights) never do, so weights they write
 *   are complete before a GEMM queued after them starts.  Kernels from other
 *   code trigger early only if they say so; for them this is plain stream
 *   order.
 */
mxfp8_status mxfp8_linear(const void* x_bf16, const uint8_t* x_q, const uint8_t* x_scale,
                          int64_t B, int64_t M, int64_t N, int64_t K, const uint8_t* w_packed,
                          const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                          void* workspace, size_t workspace_bytes, mxfp8_stream_t stream);

/*
 * mxfp8_linear_path - mxfp8_linear with the kernel path chosen by the caller
 * instead of by M: path 0 = automatic (as mxfp8_linear), 1 = small-M path
 * (weights on the MMA's M side; bf16 x quantised inside the GEMM, or a
 * pre-quantised x_q / x_scale copied into the same operand tiles), 2 = large-M
 * path with one CTA per 128 x 256 output tile (separate quantise kernel, then
 * the GEMM), 3 = large-M path with 256 x 256 tiles on CTA pairs (tcgen05
 * cta_group::2; what path 0 takes when the small-M path does not apply and
 * M > 128 or one wave of pairs holds every tile, B * ceil(N / 256) <= SMs / 2),
 * 4 = the large-M kernels chosen as path 0 chooses them, never the small-M one
 * (CTA pairs with split-K when the shape has at most 16 256 x 256 output
 * tiles, 32 when K >= 8192: each tile's K range is split over several pairs,
 * fp32 partials go to the workspace and are added in a fixed order, so the
 * result is the same on every call; this is also what the quantised hand-off
 * uses), 5 = x quantised inside the GEMM (bf16 x read once into shared
 * memory, quantised there by the same per-block rule into the MMA's operand
 * tile; no quantised copy of x in memory), one CTA per 128 x 256 output tile
 * (path 0 never takes it: on B = 16, M = N = 512, K = 7168 it measured no
 * faster than the quantise kernel plus the CTA-pair GEMM).  All paths compute
 * the same function; this exists so that tests can check each
 * on every shape.  Path 1 needs B = 1 and M <= 128; path 5 needs x_bf16,
 * N <= 512 and at most one 128 x 256 tile per SM (else MXFP8_ERR_UNSUPPORTED).
 */
mxfp8_status mxfp8_linear_path(int path, const void* x_bf16, const uint8_t* x_q,
                               const uint8_t* x_scale, int64_t B, int64_t M, int64_t N,
                               int64_t K, const uint8_t* w_packed, const uint8_t* sf_packed,
                               const void* bias_bf16, void* out_bf16, void* workspace,
                               size_t workspace_bytes, mxfp8_stream_t stream);

/*
 * mxfp8_quantize_packed - mxfp8_quantize for B batches of [M, K] rows, writing
 * the scales straight into the packed atom layout the GEMM reads (the same
 * layout mxfp8_process_weights gives weight scales; sf bytes as returned by
 * mxfp8_packed_sizes(B, M, K)).  Padding bytes of the last row tile are not
 * written.  This is the first half of mxfp8_linear on bf16 input.
 *   x_bf16 : device, [B, M, K] bf16.   x_q : device, [B, M, K] out.
 *   sfa_packed : device, packed scale atoms out.  K % 32 == 0, 16-byte aligned.
 */
mxfp8_status mxfp8_quantize_packed(const void* x_bf16, int64_t B, int64_t M, int64_t K,
                                   uint8_t* x_q, uint8_t* sfa_packed, mxfp8_stream_t stream);

/*
 * mxfp8_pack_scales - row-major E8M0 scales [B, R, K/32] -> packed atoms
 * (zero padding), for any operand; mxfp8_process_weights uses it for weight
 * scales and mxfp8_linear for pre-quantised activation scales.  scale and
 * sf_packed: device, 16-byte aligned.
 */
mxfp8_status mxfp8_pack_scales(const uint8_t* scale, int64_t B, int64_t R, int64_t K,
                               uint8_t* sf_packed, mxfp8_stream_t stream);

/*
 * mxfp8_gemm_packed - the block-scaled GEMM and epilogue alone, both operands
 * already packed: out = bf16(x_q . w^T (block-scaled) + bias).  The second half
 * of mxfp8_linear.  Requirements as for mxfp8_linear (N % 8 == 0, K % 128 == 0).
 *   x_q, sfa_packed : device, from mxfp8_quantize_packed (or mxfp8_pack_scales).
 *   w_packed, sf_packed : device, from mxfp8_process_weights.
 *   With B = 1 and up to 64 rows (up to 128 where the small-M kernel's K split
 *   leaves each CTA at most 1024 of K) the small-M kernel runs, copying the
 *   codes and scale atoms into its operand tiles, and the output is what
 *   mxfp8_linear gives for the x these operands were quantised from;
 *   otherwise the large-M kernels, which here never split K (where
 *   mxfp8_linear splits K its fp32 sums are rounded in another order).
 */
mxfp8_status mxfp8_gemm_packed(const uint8_t* x_q, const uint8_t* sfa_packed, int64_t B, int64_t M,
                               int64_t N, int64_t K, const uint8_t* w_packed,
                               const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                               mxfp8_stream_t stream);

/*
 * mxfp8_linear_quantized_out - mxfp8_linear whose output is handed on to the
 * next layer already quantised (the QuantizedActivation hand-off).
 *   Source: "AiterFlyDSLMxfp8LinearKernel.apply_weights" (aiter_flydsl page):
 *   a layer accepts its input as a QuantizedActivation (data + scale) when the
 *   previous op produced one, and then skips its own quantise step.  Here the
 *   GEMM epilogue produces it: y = bf16(x . w^T + bias), quantised by the
 *   mxfp8_quantize rule (OCP MX v1.0, section 6.3) on the same bf16 bits, so
 *   y_q / y_sf_packed are the bytes mxfp8_quantize_packed(y) would write
 *   (padding rows of the last atom tile are left as they were).  The call
 *   runs the kernels mxfp8_linear chooses and y is its output bit for bit,
 *   except at B = 1 and decode sizes where mxfp8_linear's small-M kernel
 *   splits K eight ways (N below ~2048): the hand-off splits it four ways
 *   (whole 32-column blocks per CTA), so its fp32 sums are rounded in
 *   another order.
 *   Inputs, w_packed, sf_packed, bias, workspace: as mxfp8_linear (either x
 *   form; the workspace of mxfp8_workspace_size).
 *   out_bf16    : device, [B, M, N] bf16 out, or NULL to skip the bf16 output.
 *   y_q         : device, [B, M, N] E4M3 codes out (16-byte aligned).
 *   y_sf_packed : device, packed scale atoms of (B, M, N) out, the
 *                 mxfp8_packed_sizes(B, M, N) sf bytes (16-byte aligned): the
 *                 activation-scale operand of mxfp8_gemm_packed for the next
 *                 layer (K = N).
 *   Requirements as mxfp8_linear, and N % 128 == 0 (the next layer's K;
 *   else MXFP8_ERR_UNSUPPORTED).
 */
mxfp8_status mxfp8_linear_quantized_out(const void* x_bf16, const uint8_t* x_q, const uint8_t* x_scale,
                                        int64_t B, int64_t M, int64_t N, int64_t K, const uint8_t* w_packed,
                                        const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                                        uint8_t* y_q, uint8_t* y_sf_packed, void* workspace,
                                        size_t workspace_bytes, mxfp8_stream_t stream);

/*
 * mxfp8_gemm_packed_quantized_out - mxfp8_gemm_packed with the same quantised
 * hand-off output as mxfp8_linear_quantized_out: the step of a chain of layers
 * whose input is the previous layer's y_q / y_sf_packed and whose output feeds
 * the next.  Source and arguments as those two calls (out_bf16 may be NULL;
 * N % 128 == 0); the kernel choice as mxfp8_gemm_packed's, K split at most
 * four ways on the small-M kernel.
 */
mxfp8_status mxfp8_gemm_packed_quantized_out(const uint8_t* x_q, const uint8_t* sfa_packed, int64_t B, int64_t M,
                                             int64_t N, int64_t K, const uint8_t* w_packed,
                                             const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                                             uint8_t* y_q, uint8_t* y_sf_packed, mxfp8_stream_t stream);

/*
 * Size of the fixed device scratch array used by mxfp8_linear_noalloc.
 */
#define MXFP8_NOALLOC_SCRATCH_BYTES (32ll << 20)

/*
 * mxfp8_linear_noalloc - mxfp8_linear for bf16 input, for callers that cannot
 * allocate device memory (no workspace argument).  No counterpart on the
 * source pages: their layer always allocates its quantised activation.
 *   Who needs it: a process whose GPU memory is already owned by another
 *   allocator (a serving runtime that reserves the device at start-up, where a
 *   new cudaMalloc fails or fragments that pool), or a runtime with a fixed
 *   memory plan that forbids allocation after initialisation.
 *   Scratch: a file-scope device array of MXFP8_NOALLOC_SCRATCH_BYTES (32 MiB)
 *   inside the library, held by every GPU that loads the library until the
 *   process exits.  With B = 1 and M <= 32 (or M <= 64 where the small-M
 *   kernel splits K, or M <= 128 where it splits K into ranges of at most
 *   1024) the call runs the small-M kernel, which quantises x inside the
 *   GEMM and uses no scratch; otherwise it needs
 *   round_up(B*M*K, 256) + round_up(packed scale bytes of (B, M, K), 256)
 *   bytes of it and returns MXFP8_ERR_UNSUPPORTED beyond that (e.g. M*K above
 *   ~32.5 M at B = 1).
 *   Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  Every call shares the one array, so calls
 *   that overlap on the GPU (different streams or threads) race and must be
 *   serialised by the caller.
 *   Arguments, layouts and requirements as for mxfp8_linear with x_bf16
 *   (B >= 1, N % 8 == 0, K % 128 == 0, 16-byte aligned pointers).
 */
mxfp8_status mxfp8_linear_noalloc(const void* x_bf16, int64_t B, int64_t M, int64_t N, int64_t K,
                                  const uint8_t* w_packed, const uint8_t* sf_packed,
                                  const void* bias_bf16, void* out_bf16, mxfp8_stream_t stream);

/*
 * MXFP6 weights.
 *   Source: the mxfp6 page: "MxFp6LinearLayerConfig" (weights quantised per
 *   block of 32, weight_quant_key kMxfp6E2M3Static or kMxfp6E3M2Static) and
 *   "MxFp6LinearKernel" (process_weights_after_loading, apply_weights).  The
 *   element formats are OCP MX v1.0 FP6 (section 5.3.2): E2M3 (bias 1, largest
 *   7.5, emax 2) and E3M2 (bias 3, largest 28, emax 4), with the same E8M0
 *   block scales (e = floor(log2 amax) - emax) and MXFP8 activations; the
 *   tensor cores multiply them directly (kind::mxf8f6f4).
 *   Packed FP6 weights are 3K/4 bytes per row: every 16 codes of a row are
 *   12 bytes, code i in bits [6i, 6i + 6) of the little-endian 96-bit group
 *   (25 % fewer weight bytes than E4M3).  They need K % 128 == 0 and
 *   w_packed 32-byte aligned.
 */
#define MXFP8_WFMT_E4M3 0
#define MXFP8_WFMT_E2M3 1
#define MXFP8_WFMT_E3M2 2

/*
 * mxfp8_quantize_weights - bf16 weights -> w_format codes, one per byte
 * (E4M3 bytes, or FP6 codes in the low 6 bits), and row-major E8M0 scales
 * [rows, K/32], by the rule of mxfp8_quantize with the format's emax.  A block
 * holding Inf or NaN gets scale 0xFF and codes 0x7F (E4M3) or 0x00 (FP6).
 * Pointers: device, 16-byte aligned; K % 32 == 0.
 */
mxfp8_status mxfp8_quantize_weights(const void* w_bf16, int64_t rows, int64_t K, int w_format, uint8_t* w_q,
                                    uint8_t* w_scale, mxfp8_stream_t stream);

/* mxfp8_packed_sizes for weights of w_format (FP6: 3BNK/4 weight bytes). */
mxfp8_status mxfp8_packed_sizes_fmt(int w_format, int64_t B, int64_t N, int64_t K, size_t* w_bytes,
                                    size_t* sf_bytes);

/*
 * mxfp8_process_weights_fmt - mxfp8_process_weights for w_format weights:
 * w holds one code per byte ([B, N, K], FP6 codes in the low 6 bits); for
 * FP6 the codes are packed to 6 bits (w_packed != w, mxfp8_packed_sizes_fmt
 * bytes, 32-byte aligned).  Scales as mxfp8_process_weights.
 */
mxfp8_status mxfp8_process_weights_fmt(int w_format, const uint8_t* w, const uint8_t* w_scale, int64_t B, int64_t N,
                                       int64_t K, uint8_t* w_packed, uint8_t* sf_packed, mxfp8_stream_t stream);

/*
 * mxfp8_linear_fmt - mxfp8_linear_path for weights of w_format (packed by
 * mxfp8_process_weights_fmt with the same format): the block-scaled product
 * of MXFP8 activations with MXFP6 (or MXFP8) weights.  Arguments and
 * requirements as mxfp8_linear_path.
 */
mxfp8_status mxfp8_linear_fmt(int path, int w_format, const void* x_bf16, const uint8_t* x_q,
                              const uint8_t* x_scale, int64_t B, int64_t M, int64_t N, int64_t K,
                              const uint8_t* w_packed, const uint8_t* sf_packed, const void* bias_bf16,
                              void* out_bf16, void* workspace, size_t workspace_bytes, mxfp8_stream_t stream);

/*
 * Persistable packed weights.
 *   Source: the Mxfp8LinearKernel page: supports_pre_processed_weights and the
 *   weight-cache daemon that hands weights, already processed, to later
 *   processes, which use them as they are.  The output of
 *   mxfp8_process_weights depends only on (B, N, K) and on this library's
 *   layout, so it can be stored once and reloaded without repacking.
 *   A blob is a 128-byte header (magic "MXFP8PW1", format version, layout id,
 *   flags, B, N, K, payload sizes, an FNV-1a 64 checksum of the payload and
 *   one of the header; integers little-endian) followed by the w_packed bytes
 *   and the sf_packed bytes.  These calls work on HOST memory only (no CUDA
 *   call, no device memory): the caller copies the payloads between host and
 *   device (cudaMemcpy or torch).
 */
#define MXFP8_BLOB_HEADER_BYTES 128

/* Bytes of the blob for B batches of an [N, K] layer of w_format weights
 * (header + payloads). */
mxfp8_status mxfp8_blob_size(int64_t B, int64_t N, int64_t K, int w_format, size_t* bytes);

/*
 * mxfp8_weights_serialize - write a blob.
 *   w_packed, sf_packed : host, the mxfp8_packed_sizes_fmt(w_format, B, N, K)
 *                         bytes of each (as mxfp8_process_weights[_fmt] wrote
 *                         them, copied to host).
 *   w_format            : MXFP8_WFMT_*, stored as the layout id (so a reader
 *                         cannot take packed FP6 bytes for E4M3).
 *   batched             : 1 if the layer's weights are [B, N, K] (bmm), else 0;
 *                         stored so that a reader restores the same shapes.
 *   blob                : host, >= mxfp8_blob_size(B, N, K) bytes, written.
 *   MXFP8_ERR_INVALID_ARG on a null pointer, a bad shape or a short blob.
 */
mxfp8_status mxfp8_weights_serialize(const uint8_t* w_packed, const uint8_t* sf_packed, int64_t B,
                                     int64_t N, int64_t K, int w_format, int batched, uint8_t* blob,
                                     size_t blob_bytes);

/*
 * mxfp8_weights_deserialize - check a blob and locate its payloads.
 *   blob, blob_bytes : host, the bytes written by mxfp8_weights_serialize.
 *   B, N, K, w_format, batched : out, the stored shape and weight format.
 *   w_offset, sf_offset : out, byte offsets of the w_packed and sf_packed
 *                         payloads inside blob (16-byte aligned offsets; the
 *                         sizes are those of mxfp8_packed_sizes_fmt).
 *   MXFP8_ERR_INVALID_ARG: null pointer, not a blob, truncated, or either
 *   checksum wrong (corrupted).  MXFP8_ERR_UNSUPPORTED: written with another
 *   format version or layout (repack with mxfp8_process_weights instead).
 *   Nothing is written to the outputs unless the blob is valid.
 */
mxfp8_status mxfp8_weights_deserialize(const uint8_t* blob, size_t blob_bytes, int64_t* B, int64_t* N,
                                       int64_t* K, int* w_format, int* batched, size_t* w_offset,
                                       size_t* sf_offset);

/*
 * mxfp8_check - synchronise `stream`, then read and clear the device status
 * word of the current device.  Returns MXFP8_ERR_TIMEOUT if a bounded wait in
 * any kernel of this library ran out since the last check, MXFP8_ERR_CUDA if
 * the stream reports an error, else MXFP8_OK.
 */
mxfp8_status mxfp8_check(mxfp8_stream_t stream);

/*
 * mxfp8_debug_expire_wait - launch one tiny kernel whose mbarrier wait can
 * never complete (nothing arrives), bounded by timeout_ns nanoseconds
 * (1e3 <= timeout_ns <= 1e10).  The kernel records the expiry in the status
 * word and returns, so that tests can see the timeout path work end to end
 * (mxfp8_check then returns MXFP8_ERR_TIMEOUT).  No counterpart on the pages.
 */
mxfp8_status mxfp8_debug_expire_wait(uint64_t timeout_ns, mxfp8_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_H */
