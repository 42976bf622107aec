// api.cu - the C ABI of libmxfp8.so (declared in include/mxfp8.h).
//
// Host-side only: argument checks (all before any launch), workspace carving,
// and the choice between the two linear paths.  The pages' kernel interface
// ("Mxfp8LinearKernel": is_supported / can_implement / process_weights_after_
// loading / apply_weights) maps onto it as: is_supported -> MXFP8_ERR_ARCH,
// can_implement -> MXFP8_ERR_UNSUPPORTED, process_weights_after_loading ->
// mxfp8_process_weights, apply_weights -> mxfp8_linear.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/mxfp8.h"
#include "mx_kernels.h"
#include "mx_layout.cuh"

namespace {

thread_local std::string g_last_error;

mxfp8_status fail(mxfp8_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mxfp8_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MXFP8_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  int major = 0, minor = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Current device, checked to be sm_103.  Returns MXFP8_OK and fills *sms.
mxfp8_status current_device(int* sms) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MXFP8_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ok) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ok = true;
  }
  if (d.major != 10 || d.minor != 3)
    return fail(MXFP8_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                d.major, d.minor);
  *sms = d.sms;
  return MXFP8_OK;
}

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

constexpr int kSmallM = mx::kDecodeMaxM;  // largest M the small-M kernel takes

struct WsLayout {
  int64_t xq_off, xq_bytes, sfa_off, sfa_bytes, part_off, part_bytes, total;
};

// Workspace of a large-M call: quantised activations (bf16 input only), their
// packed scales, then the split-K partials (fp32 [splits * B][M][N]) when the
// shape is split.
WsLayout prefill_workspace(int64_t B, int64_t M, int64_t N, int64_t K, bool quantized, int splits) {
  WsLayout w;
  w.xq_off = 0;
  w.xq_bytes = quantized ? 0 : round_up(B * M * K, 256);
  w.sfa_off = w.xq_bytes;
  w.sfa_bytes = round_up(mx::sf_packed_bytes(B, M, K), 256);
  w.part_off = w.sfa_off + w.sfa_bytes;
  w.part_bytes = splits > 1 ? round_up(static_cast<int64_t>(splits) * B * M * N * 4, 256) : 0;
  w.total = w.part_off + w.part_bytes;
  return w;
}

// The quantise and repack kernels index 32-element blocks and 4-byte packed
// scale words with 32-bit integers: B*R*(K/32) blocks and the packed scale
// words of (B, R, K) must each fit in 31 bits.  Sizes are checked for range
// first, so the products below cannot overflow 64 bits.
mxfp8_status check_block_count(int64_t B, int64_t R, int64_t K, const char* what) {
  if (B > (1ll << 20) || R > (1ll << 31) || K > (1ll << 30) || B * R > (1ll << 31) ||
      B * R * (K / 32) > mx::kMaxBlocks32 || mx::sf_packed_bytes(B, R, K) / 4 > mx::kMaxBlocks32)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "%s: B=%lld R=%lld K=%lld has more than 2^31 - 1 scale blocks; split the call",
                what, (long long)B, (long long)R, (long long)K);
  return MXFP8_OK;
}

mxfp8_status check_weights_args(const void* w, const void* ws, int64_t B, int64_t N, int64_t K) {
  if (w == nullptr || ws == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null weight pointer");
  if (B < 1 || N < 1 || K < 1) return fail(MXFP8_ERR_INVALID_ARG, "B=%lld N=%lld K=%lld", (long long)B, (long long)N, (long long)K);
  if (K % 32 != 0) return fail(MXFP8_ERR_INVALID_ARG, "K=%lld is not a multiple of 32", (long long)K);
  if (!aligned(w, 16) || !aligned(ws, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "weight and scale pointers must be 16-byte aligned");
  return check_block_count(B, N, K, "scales");
}

mxfp8_status check_gemm_args(int64_t B, int64_t M, int64_t N, int64_t K) {
  if (B < 1 || M < 0 || N < 1 || K < 1)
    return fail(MXFP8_ERR_INVALID_ARG, "B=%lld M=%lld N=%lld K=%lld", (long long)B, (long long)M,
                (long long)N, (long long)K);
  if (K % 32 != 0) return fail(MXFP8_ERR_INVALID_ARG, "K=%lld is not a multiple of 32", (long long)K);
  if (K % 128 != 0)
    return fail(MXFP8_ERR_UNSUPPORTED, "K=%lld: this library needs K %% 128 == 0", (long long)K);
  if (N % 8 != 0)
    return fail(MXFP8_ERR_UNSUPPORTED, "N=%lld: this library needs N %% 8 == 0", (long long)N);
  if (B * M > (1ll << 31) || N > (1ll << 30) || K > (1ll << 30))
    return fail(MXFP8_ERR_UNSUPPORTED, "problem too large");
  if (M > 0) {
    mxfp8_status st = check_block_count(B, M, K, "activations");
    if (st != MXFP8_OK) return st;
  }
  return check_block_count(B, N, K, "weights");
}

}  // namespace

namespace mx {

void set_last_error(const char* msg) { g_last_error = msg; }

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace mx

extern "C" {

const char* mxfp8_last_error(void) { return g_last_error.c_str(); }

int mxfp8_version(void) { return 1; }

mxfp8_status mxfp8_quantize(const void* x_bf16, int64_t rows, int64_t K, uint8_t* x_q,
                            uint8_t* x_scale, mxfp8_stream_t stream) {
  if (rows < 0 || K < 1) return fail(MXFP8_ERR_INVALID_ARG, "rows=%lld K=%lld", (long long)rows, (long long)K);
  if (K % 32 != 0) return fail(MXFP8_ERR_INVALID_ARG, "K=%lld is not a multiple of 32", (long long)K);
  if (rows == 0) return MXFP8_OK;
  if (x_bf16 == nullptr || x_q == nullptr || x_scale == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x_bf16, 16) || !aligned(x_q, 16) || !aligned(x_scale, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "x_bf16, x_q and x_scale must be 16-byte aligned");
  mxfp8_status st = check_block_count(1, rows, K, "mxfp8_quantize");
  if (st != MXFP8_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaError_t e = mx::launch_quantize(x_bf16, rows, K, x_q, x_scale, false, 1, rows, sms,
                                      reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_packed_sizes(int64_t B, int64_t N, int64_t K, size_t* w_bytes, size_t* sf_bytes) {
  if (w_bytes == nullptr || sf_bytes == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  if (B < 1 || N < 1 || K < 1 || K % 32 != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "B=%lld N=%lld K=%lld", (long long)B, (long long)N, (long long)K);
  *w_bytes = static_cast<size_t>(B * N * K);
  *sf_bytes = static_cast<size_t>(mx::sf_packed_bytes(B, N, K));
  return MXFP8_OK;
}

mxfp8_status mxfp8_process_weights(const uint8_t* w, const uint8_t* w_scale, int64_t B, int64_t N,
                                   int64_t K, uint8_t* w_packed, uint8_t* sf_packed,
                                   mxfp8_stream_t stream) {
  mxfp8_status st = check_weights_args(w, w_scale, B, N, K);
  if (st != MXFP8_OK) return st;
  if (w_packed == nullptr || sf_packed == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  if (!aligned(w_packed, 16) || !aligned(sf_packed, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "w_packed and sf_packed must be 16-byte aligned");
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (w_packed != w) {
    cudaError_t e = cudaMemcpyAsync(w_packed, w, static_cast<size_t>(B * N * K), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "weight copy");
  }
  cudaError_t e = mx::launch_sf_pack(w_scale, B, N, K, sf_packed, sms, s, false);
  if (e != cudaSuccess) return cuda_fail(e, "scale repack launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_unpack_scales(const uint8_t* sf_packed, int64_t B, int64_t N, int64_t K,
                                 uint8_t* w_scale, mxfp8_stream_t stream) {
  mxfp8_status st = check_weights_args(sf_packed, w_scale, B, N, K);
  if (st != MXFP8_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaError_t e = mx::launch_sf_unpack(sf_packed, B, N, K, w_scale, sms,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scale unpack launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_workspace_size(int64_t B, int64_t M, int64_t N, int64_t K, int x_is_quantized,
                                  size_t* bytes) {
  if (bytes == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  if (B < 1 || M < 0 || N < 1 || K < 1 || K % 32 != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "B=%lld M=%lld N=%lld K=%lld", (long long)B, (long long)M,
                (long long)N, (long long)K);
  if (B * M > (1ll << 31) || N > (1ll << 30) || K > (1ll << 30))
    return fail(MXFP8_ERR_UNSUPPORTED, "problem too large");
  *bytes = static_cast<size_t>(prefill_workspace(B, M, N, K, x_is_quantized != 0, mx::splitk_splits(B, M, N, K)).total);
  return MXFP8_OK;
}

}  // extern "C"

namespace {

// The outputs of a linear call: the bf16 result and/or its MXFP8 quantisation
// for the next layer (codes [B, M, N] + packed scale atoms of (B, M, N)).
struct LinearOut {
  void* out_bf16;
  uint8_t* y_q;
  uint8_t* y_sf;
};

mxfp8_status check_linear_out(const LinearOut& o, int64_t B, int64_t M, int64_t N) {
  const bool hand_off = o.y_q != nullptr || o.y_sf != nullptr;
  if (hand_off && (o.y_q == nullptr || o.y_sf == nullptr))
    return fail(MXFP8_ERR_INVALID_ARG, "y_q and y_sf_packed must both be given");
  if (o.out_bf16 == nullptr && !hand_off) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  if ((o.out_bf16 != nullptr && !aligned(o.out_bf16, 16)) || (hand_off && (!aligned(o.y_q, 16) || !aligned(o.y_sf, 16))))
    return fail(MXFP8_ERR_INVALID_ARG, "output pointers must be 16-byte aligned");
  if (hand_off && N % 128 != 0)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "N=%lld: the quantised output feeds a layer with K = N, which needs N %% 128 == 0", (long long)N);
  if (hand_off && M > 0) return check_block_count(B, M, N, "quantised output");
  return MXFP8_OK;
}

mxfp8_status check_wfmt(int w_format) {
  if (w_format != MXFP8_WFMT_E4M3 && w_format != MXFP8_WFMT_E2M3 && w_format != MXFP8_WFMT_E3M2)
    return fail(MXFP8_ERR_INVALID_ARG, "w_format=%d", w_format);
  return MXFP8_OK;
}

mxfp8_status linear_impl(int path, const void* x_bf16, const uint8_t* x_q, const uint8_t* x_scale, int64_t B,
                         int64_t M, int64_t N, int64_t K, const uint8_t* w_packed, const uint8_t* sf_packed,
                         const void* bias_bf16, const LinearOut& o, void* workspace, size_t workspace_bytes,
                         mxfp8_stream_t stream, int w_format = MXFP8_WFMT_E4M3) {
  if (path < 0 || path > 5) return fail(MXFP8_ERR_INVALID_ARG, "path=%d", path);
  if (check_wfmt(w_format) != MXFP8_OK) return MXFP8_ERR_INVALID_ARG;
  {
    mxfp8_status ck = check_gemm_args(B, M, N, K);
    if (ck != MXFP8_OK) return ck;
  }
  if (M == 0) return MXFP8_OK;  // nothing to read or write; pointers may be null
  const bool have_x = x_bf16 != nullptr;
  const bool have_q = x_q != nullptr || x_scale != nullptr;
  if (have_x == have_q)
    return fail(MXFP8_ERR_INVALID_ARG, "pass exactly one of x_bf16 or (x_q, x_scale)");
  if (have_q && (x_q == nullptr || x_scale == nullptr))
    return fail(MXFP8_ERR_INVALID_ARG, "x_q and x_scale must both be given");
  if (w_packed == nullptr || sf_packed == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "null weight pointer");
  {
    mxfp8_status ck = check_linear_out(o, B, M, N);
    if (ck != MXFP8_OK) return ck;
  }
  if (!aligned(w_packed, 16) || !aligned(sf_packed, 16) ||
      (have_x && !aligned(x_bf16, 16)) || (have_q && (!aligned(x_q, 16) || !aligned(x_scale, 16))) ||
      (bias_bf16 != nullptr && !aligned(bias_bf16, 16)))
    return fail(MXFP8_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (w_format != MXFP8_WFMT_E4M3 && !aligned(w_packed, 32))
    return fail(MXFP8_ERR_INVALID_ARG, "packed FP6 weights must be 32-byte aligned");
  int sms = 0;
  mxfp8_status st = current_device(&sms);
  if (st != MXFP8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* out_bf16 = o.out_bf16;

  // The small-M kernel (every threshold below measured in CUDA graphs of
  // back-to-back calls):
  //  * quantises its output for the hand-off with K split at most four ways
  //    (a warp then holds each 32-column block; where it would split eight
  //    ways the hand-off splits four, so its sums round in another order);
  //  * up to 32 rows, quantises bf16 x inside every CTA;
  //  * from 33 to 64 rows of bf16 x, does so only while each CTA's K range is
  //    short (K split, K / S <= 1024: N = K = 4096, M = 48 / 64 9.0 / 9.5 us);
  //    otherwise path 0 quantises x once into the workspace and the kernel,
  //    launched behind the quantiser's early trigger, copies the codes
  //    (N = 14336, K = 4096: 18.3 / 18.5 us against 23.0 / 23.2 on CTA pairs
  //    and 25.1 / 25.0 re-quantising in every CTA; N = 4096, K = 14336:
  //    18.0 / 19.2 against 22.7 / 23.1 us re-quantising); with a workspace
  //    below the documented size it re-quantises instead (the same bytes);
  //  * copies a pre-quantised x, up to 64 rows (N = 14336, M = 48 / 64:
  //    19.6 / 19.9 us against 21.4 / 21.7 on CTA pairs);
  //  * from 65 to 128 rows (its 128-token shape), serves only where the K
  //    split leaves each CTA a short K range (K / S <= 1024), bf16 x
  //    quantised once and copied: N = K = 4096, M = 65 / 96 / 128
  //    12.0 / 12.6 / 14.1 us (pre-quantised 9.8 / 10.4 / 10.8) against
  //    15.4 / 16.1 / 16.4 (15.0 / 15.8 / 16.4) on split-K CTA pairs; with
  //    longer K ranges (N = 14336 unsplit, or K = 14336) it took 27-33 us
  //    against 22-25 and the CTA pairs stay.
  const int dec_splits = (M > 32 && M <= kSmallM) ? mx::decode_k_splits(M, N, K, sms) : 1;
  const bool short_k = dec_splits >= 2 && K / dec_splits <= 1024;  // each CTA's K range
  const bool wide_ok = M > 64 && M <= kSmallM && short_k;
  const WsLayout qws = prefill_workspace(1, M, N, K, false, 1);
  const bool hand_ok = o.y_q == nullptr || (B == 1 && M <= kSmallM);
  const bool copy_route = path == 0 && have_x && B == 1 && M > 32 && hand_ok &&
                          ((M <= 64 && !short_k) || wide_ok) && workspace != nullptr && aligned(workspace, 256) &&
                          static_cast<int64_t>(workspace_bytes) >= qws.total;
  const bool small_ok = B == 1 && M <= kSmallM && hand_ok &&
                        (path == 1 || M <= 32 || (M <= 64 && (have_q || copy_route || dec_splits >= 2)) || wide_ok);
  if (path == 1 && !small_ok)
    return fail(MXFP8_ERR_UNSUPPORTED, "the small-M path needs B == 1, M <= %d and no quantised output", kSmallM);
  if (path == 1 || (path == 0 && small_ok)) {
    mx::DecodeProblem p{x_bf16, w_packed, sf_packed, bias_bf16, out_bf16, M, N, K, w_format};
    p.xq = x_q;
    p.xs = x_scale;
    p.yq = o.y_q;
    p.ysf = o.y_sf;
    if (copy_route) {
      uint8_t* wsb = static_cast<uint8_t*>(workspace);
      cudaError_t e = mx::launch_quantize(x_bf16, M, K, wsb + qws.xq_off, wsb + qws.sfa_off, false, 1, M, sms, s,
                                          true);
      if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
      p.x = nullptr;
      p.xq = wsb + qws.xq_off;
      p.xs = wsb + qws.sfa_off;
    }
    const char* msg = "";
    cudaError_t e = mx::launch_gemm_decode(p, sms, s, &msg);
    if (e != cudaSuccess) return cuda_fail(e, msg);
    return MXFP8_OK;
  }

  // path 5: x quantised inside the GEMM (no quantised copy of x in memory),
  // for bf16 x whose 128 x 256 output tiles fit on the GPU at once and whose
  // rows at most two column tiles share (N <= 512); not for the hand-off.
  // Path 0 does not take it: on the batched B = 16, M = N = 512, K = 7168
  // layer it measured 63.6 us against 63.5 us for quantise + CTA-pair GEMM.
  const int64_t fq_tiles = mx::fused_quantize_tiles(B, M, N);
  const bool fused_ok = have_x && o.y_q == nullptr && out_bf16 != nullptr && N <= 512 && N % 8 == 0 &&
                        fq_tiles <= sms;
  if (path == 5 && !fused_ok)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "the fused-quantise path needs bf16 x, a bf16 output, N <= 512, N %% 8 == 0 and at most %d "
                "tiles of 128 x 256",
                sms);
  if (path == 5) {
    mx::FusedProblem p{x_bf16, w_packed, sf_packed, bias_bf16, out_bf16, B, M, N, K, w_format};
    const char* msg = "";
    cudaError_t e = mx::launch_gemm_fq(p, sms, s, &msg);
    if (e != cudaSuccess) return cuda_fail(e, msg);
    return MXFP8_OK;
  }

  // paths 0 and 4 split K over CTA pairs when the shape has few output tiles
  const int splits = (path == 0 || path == 4) ? mx::splitk_splits(B, M, N, K) : 1;
  const WsLayout ws = prefill_workspace(B, M, N, K, have_q, splits);
  if (static_cast<int64_t>(workspace_bytes) < ws.total)
    return fail(MXFP8_ERR_INVALID_ARG, "workspace has %zu bytes, needs %lld", workspace_bytes,
                (long long)ws.total);
  if (workspace == nullptr || !aligned(workspace, 256))
    return fail(MXFP8_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  uint8_t* sfa = wsb + ws.sfa_off;
  mx::GemmProblem p{have_x ? wsb + ws.xq_off : x_q, w_packed, sfa, sf_packed, bias_bf16, out_bf16, B, M, N, K,
                    path == 3 ? 2 : (path == 2 ? 1 : 0), o.y_q, o.y_sf, w_format};
  if (splits > 1) {
    p.part = reinterpret_cast<float*>(wsb + ws.part_off);
    p.splits = splits;
  }
  cudaError_t e;
  if (have_x) {
    e = mx::launch_quantize(x_bf16, B * M, K, wsb + ws.xq_off, sfa, true, B, M, sms, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  } else if (mx::gemm_prefill_uses_pair(p, sms)) {
    // the CTA-pair kernel's scale writers read the row-major x_scale
    // themselves: no repack launch
    p.sfa = x_scale;
    p.sfa_rowmajor = 1;
  } else {
    e = mx::launch_sf_pack(x_scale, B, M, K, sfa, sms, s, true);
    if (e != cudaSuccess) return cuda_fail(e, "activation scale repack launch");
  }
  const char* msg = "";
  e = mx::launch_gemm_prefill(p, sms, s, &msg);
  if (e != cudaSuccess) return cuda_fail(e, msg);
  return MXFP8_OK;
}

mxfp8_status gemm_packed_impl(const uint8_t* x_q, const uint8_t* sfa_packed, int64_t B, int64_t M, int64_t N,
                              int64_t K, const uint8_t* w_packed, const uint8_t* sf_packed, const void* bias_bf16,
                              const LinearOut& o, mxfp8_stream_t stream) {
  mxfp8_status st = check_gemm_args(B, M, N, K);
  if (st != MXFP8_OK) return st;
  if (x_q == nullptr || sfa_packed == nullptr || w_packed == nullptr || sf_packed == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "null pointer");
  if ((st = check_linear_out(o, B, M, N)) != MXFP8_OK) return st;
  if (!aligned(x_q, 16) || !aligned(sfa_packed, 16) || !aligned(w_packed, 16) || !aligned(sf_packed, 16) ||
      (bias_bf16 != nullptr && !aligned(bias_bf16, 16)))
    return fail(MXFP8_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (M == 0) return MXFP8_OK;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  // Decode-sized operands (B = 1): the small-M kernel copies the codes and
  // the scale bytes from their atoms, on the shapes where mxfp8_linear gives
  // it a pre-quantised x (up to 64 rows; up to 128 where its K split leaves
  // each CTA at most 1024 of K); a hand-off as in mxfp8_linear_quantized_out.
  if (B == 1 && M <= kSmallM) {
    const int S = M > 64 ? mx::decode_k_splits(M, N, K, sms) : 0;
    if (M <= 64 || (S >= 2 && K / S <= 1024)) {
      mx::DecodeProblem dp{nullptr, w_packed, sf_packed, bias_bf16, o.out_bf16, M, N, K};
      dp.xq = x_q;
      dp.xs = sfa_packed;
      dp.xs_packed = 1;
      dp.yq = o.y_q;
      dp.ysf = o.y_sf;
      const char* msg = "";
      cudaError_t e = mx::launch_gemm_decode(dp, sms, reinterpret_cast<cudaStream_t>(stream), &msg);
      if (e != cudaSuccess) return cuda_fail(e, msg);
      return MXFP8_OK;
    }
  }
  mx::GemmProblem p{x_q, w_packed, sfa_packed, sf_packed, bias_bf16, o.out_bf16, B, M, N, K, 0, o.y_q, o.y_sf};
  const char* msg = "";
  cudaError_t e = mx::launch_gemm_prefill(p, sms, reinterpret_cast<cudaStream_t>(stream), &msg);
  if (e != cudaSuccess) return cuda_fail(e, msg);
  return MXFP8_OK;
}

}  // namespace

extern "C" {

mxfp8_status mxfp8_linear_path(int path, const void* x_bf16, const uint8_t* x_q,
                               const uint8_t* x_scale, int64_t B, int64_t M, int64_t N, int64_t K,
                               const uint8_t* w_packed, const uint8_t* sf_packed,
                               const void* bias_bf16, void* out_bf16, void* workspace,
                               size_t workspace_bytes, mxfp8_stream_t stream) {
  if (out_bf16 == nullptr && M != 0) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  return linear_impl(path, x_bf16, x_q, x_scale, B, M, N, K, w_packed, sf_packed, bias_bf16,
                     LinearOut{out_bf16, nullptr, nullptr}, workspace, workspace_bytes, stream);
}

mxfp8_status mxfp8_linear_fmt(int path, int w_format, const void* x_bf16, const uint8_t* x_q,
                              const uint8_t* x_scale, int64_t B, int64_t M, int64_t N, int64_t K,
                              const uint8_t* w_packed, const uint8_t* sf_packed, const void* bias_bf16,
                              void* out_bf16, void* workspace, size_t workspace_bytes, mxfp8_stream_t stream) {
  if (out_bf16 == nullptr && M != 0) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  return linear_impl(path, x_bf16, x_q, x_scale, B, M, N, K, w_packed, sf_packed, bias_bf16,
                     LinearOut{out_bf16, nullptr, nullptr}, workspace, workspace_bytes, stream, w_format);
}

mxfp8_status mxfp8_quantize_weights(const void* w_bf16, int64_t rows, int64_t K, int w_format, uint8_t* w_q,
                                    uint8_t* w_scale, mxfp8_stream_t stream) {
  if (check_wfmt(w_format) != MXFP8_OK) return MXFP8_ERR_INVALID_ARG;
  if (rows < 0 || K < 1 || K % 32 != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "rows=%lld K=%lld (K %% 32 == 0)", (long long)rows, (long long)K);
  if (rows == 0) return MXFP8_OK;
  if (w_bf16 == nullptr || w_q == nullptr || w_scale == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null pointer");
  if (!aligned(w_bf16, 16) || !aligned(w_q, 16) || !aligned(w_scale, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  mxfp8_status st = check_block_count(1, rows, K, "mxfp8_quantize_weights");
  if (st != MXFP8_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaError_t e = mx::launch_quantize_weights(w_bf16, rows, K, w_format, w_q, w_scale, sms,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "weight quantize launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_packed_sizes_fmt(int w_format, int64_t B, int64_t N, int64_t K, size_t* w_bytes,
                                    size_t* sf_bytes) {
  if (check_wfmt(w_format) != MXFP8_OK) return MXFP8_ERR_INVALID_ARG;
  mxfp8_status st = mxfp8_packed_sizes(B, N, K, w_bytes, sf_bytes);
  if (st != MXFP8_OK) return st;
  if (w_format != MXFP8_WFMT_E4M3) {
    if (K % 128 != 0)
      return fail(MXFP8_ERR_UNSUPPORTED, "K=%lld: packed FP6 weights need K %% 128 == 0", (long long)K);
    *w_bytes = static_cast<size_t>(B * N * K / 4 * 3);
  }
  return MXFP8_OK;
}

mxfp8_status mxfp8_process_weights_fmt(int w_format, const uint8_t* w, const uint8_t* w_scale, int64_t B, int64_t N,
                                       int64_t K, uint8_t* w_packed, uint8_t* sf_packed, mxfp8_stream_t stream) {
  if (check_wfmt(w_format) != MXFP8_OK) return MXFP8_ERR_INVALID_ARG;
  if (w_format == MXFP8_WFMT_E4M3) return mxfp8_process_weights(w, w_scale, B, N, K, w_packed, sf_packed, stream);
  mxfp8_status st = check_weights_args(w, w_scale, B, N, K);
  if (st != MXFP8_OK) return st;
  if (K % 128 != 0)
    return fail(MXFP8_ERR_UNSUPPORTED, "K=%lld: packed FP6 weights need K %% 128 == 0", (long long)K);
  if (w_packed == nullptr || sf_packed == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  if (!aligned(w_packed, 32) || !aligned(sf_packed, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "w_packed must be 32-byte and sf_packed 16-byte aligned");
  if (B * N * K / 16 > mx::kMaxBlocks32) return fail(MXFP8_ERR_UNSUPPORTED, "too many FP6 weights for one call");
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = mx::launch_fp6_pack(w, B * N * K, w_packed, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "FP6 repack launch");
  e = mx::launch_sf_pack(w_scale, B, N, K, sf_packed, sms, s, false);
  if (e != cudaSuccess) return cuda_fail(e, "scale repack launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_linear_quantized_out(const void* x_bf16, const uint8_t* x_q, const uint8_t* x_scale,
                                        int64_t B, int64_t M, int64_t N, int64_t K, const uint8_t* w_packed,
                                        const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                                        uint8_t* y_q, uint8_t* y_sf_packed, void* workspace,
                                        size_t workspace_bytes, mxfp8_stream_t stream) {
  if (M != 0 && (y_q == nullptr || y_sf_packed == nullptr))
    return fail(MXFP8_ERR_INVALID_ARG, "y_q and y_sf_packed are required");
  return linear_impl(0, x_bf16, x_q, x_scale, B, M, N, K, w_packed, sf_packed, bias_bf16,
                     LinearOut{out_bf16, y_q, y_sf_packed}, workspace, workspace_bytes, stream);
}

mxfp8_status mxfp8_gemm_packed_quantized_out(const uint8_t* x_q, const uint8_t* sfa_packed, int64_t B, int64_t M,
                                             int64_t N, int64_t K, const uint8_t* w_packed,
                                             const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                                             uint8_t* y_q, uint8_t* y_sf_packed, mxfp8_stream_t stream) {
  if (M != 0 && (y_q == nullptr || y_sf_packed == nullptr))
    return fail(MXFP8_ERR_INVALID_ARG, "y_q and y_sf_packed are required");
  return gemm_packed_impl(x_q, sfa_packed, B, M, N, K, w_packed, sf_packed, bias_bf16,
                          LinearOut{out_bf16, y_q, y_sf_packed}, stream);
}

mxfp8_status mxfp8_linear(const void* x_bf16, const uint8_t* x_q, const uint8_t* x_scale, int64_t B,
                          int64_t M, int64_t N, int64_t K, const uint8_t* w_packed,
                          const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                          void* workspace, size_t workspace_bytes, mxfp8_stream_t stream) {
  return mxfp8_linear_path(0, x_bf16, x_q, x_scale, B, M, N, K, w_packed, sf_packed, bias_bf16,
                           out_bf16, workspace, workspace_bytes, stream);
}

mxfp8_status mxfp8_quantize_packed(const void* x_bf16, int64_t B, int64_t M, int64_t K,
                                   uint8_t* x_q, uint8_t* sfa_packed, mxfp8_stream_t stream) {
  if (B < 1 || M < 0 || K < 1 || K % 32 != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "B=%lld M=%lld K=%lld", (long long)B, (long long)M, (long long)K);
  if (M == 0) return MXFP8_OK;
  if (x_bf16 == nullptr || x_q == nullptr || sfa_packed == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x_bf16, 16) || !aligned(x_q, 16) || !aligned(sfa_packed, 16))
    return fail(MXFP8_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  mxfp8_status st = check_block_count(B, M, K, "mxfp8_quantize_packed");
  if (st != MXFP8_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaError_t e = mx::launch_quantize(x_bf16, B * M, K, x_q, sfa_packed, true, B, M, sms,
                                      reinterpret_cast<cudaStream_t>(stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_pack_scales(const uint8_t* scale, int64_t B, int64_t R, int64_t K,
                               uint8_t* sf_packed, mxfp8_stream_t stream) {
  mxfp8_status st = check_weights_args(scale, sf_packed, B, R, K);  // both pointers 16-byte aligned
  if (st != MXFP8_OK) return st;
  int sms = 0;
  if ((st = current_device(&sms)) != MXFP8_OK) return st;
  cudaError_t e = mx::launch_sf_pack(scale, B, R, K, sf_packed, sms, reinterpret_cast<cudaStream_t>(stream),
                                     false);
  if (e != cudaSuccess) return cuda_fail(e, "scale repack launch");
  return MXFP8_OK;
}

mxfp8_status mxfp8_gemm_packed(const uint8_t* x_q, const uint8_t* sfa_packed, int64_t B, int64_t M,
                               int64_t N, int64_t K, const uint8_t* w_packed,
                               const uint8_t* sf_packed, const void* bias_bf16, void* out_bf16,
                               mxfp8_stream_t stream) {
  if (out_bf16 == nullptr && M != 0) return fail(MXFP8_ERR_INVALID_ARG, "null output pointer");
  return gemm_packed_impl(x_q, sfa_packed, B, M, N, K, w_packed, sf_packed, bias_bf16,
                          LinearOut{out_bf16, nullptr, nullptr}, stream);
}

mxfp8_status mxfp8_check(mxfp8_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int s1 = 0, s2 = 0, s3 = 0, s4 = 0, s5 = 0, s6 = 0;
  if ((e = mx::take_status_quantize(&s1)) != cudaSuccess ||
      (e = mx::take_status_gemm(&s2)) != cudaSuccess ||
      (e = mx::take_status_decode(&s3)) != cudaSuccess ||
      (e = mx::take_status_pair(&s4)) != cudaSuccess ||
      (e = mx::take_status_fq(&s6)) != cudaSuccess ||
      (e = mx::take_status_debug(&s5)) != cudaSuccess)
    return cuda_fail(e, "status word read");
  if ((s1 | s2 | s3 | s4 | s5 | s6) & 1u) return fail(MXFP8_ERR_TIMEOUT, "a bounded in-kernel wait ran out");
  return MXFP8_OK;
}

mxfp8_status mxfp8_debug_expire_wait(uint64_t timeout_ns, mxfp8_stream_t stream) {
  if (timeout_ns < 1000 || timeout_ns > 10000000000ull)
    return fail(MXFP8_ERR_INVALID_ARG, "timeout_ns=%llu out of [1e3, 1e10]", (unsigned long long)timeout_ns);
  int sms = 0;
  mxfp8_status st = current_device(&sms);
  if (st != MXFP8_OK) return st;
  cudaError_t e = mx::launch_expire_wait(timeout_ns, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "debug kernel launch");
  return MXFP8_OK;
}

}  // extern "C"
