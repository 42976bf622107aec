// noalloc.cu - mxfp8_linear_noalloc: the bf16-input linear layer for callers
// that cannot allocate device memory.
//
// mxfp8_linear needs a workspace (the quantised activations and their packed
// scales) that the caller allocates.  Some callers cannot: a serving runtime
// that reserved the whole GPU for its own pool at start-up, where a fresh
// cudaMalloc fails or fragments that pool, or a runtime with a fixed memory plan
// that forbids any allocation after initialisation.  This entry point keeps its
// scratch in a fixed-size array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoallocScratchBytes for it until the process exits.  Host code
// cannot use the array's name as a device address (on the host it names a
// stand-in object), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, and passes the pointer to
// the kernels.  All calls share the one array: calls that overlap on the GPU
// (other streams, other threads) race on it and must be serialised by the
// caller.  Nothing in it needs to start at zero: every scratch byte the stored
// outputs depend on is written by the same call before the GEMM reads it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mxfp8.h"
#include "mx_kernels.h"
#include "mx_layout.cuh"

namespace {

constexpr int64_t kNoallocScratchBytes = MXFP8_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

mxfp8_status fail(mxfp8_status st, const char* msg) {
  mx::set_last_error(msg);
  return st;
}

// Device address of the scratch array and SM count for the current device,
// looked up once per device (with that device current).
mxfp8_status scratch_for_current_device(uint8_t** ptr, int* sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: cudaGetDevice failed");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: cudaDeviceGetAttribute failed");
    if (major != 10 || minor != 3)
      return fail(MXFP8_ERR_ARCH, "mxfp8_linear_noalloc: the current device is not sm_103");
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: cudaGetSymbolAddress of the scratch array failed");
    g_scratch_ptr[dev] = p;
    g_sms[dev] = n;
  }
  *ptr = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  *sms = g_sms[dev];
  return MXFP8_OK;
}

}  // namespace

extern "C" mxfp8_status mxfp8_linear_noalloc(const void* x_bf16, int64_t B, int64_t M, int64_t N,
                                             int64_t K, const uint8_t* w_packed,
                                             const uint8_t* sf_packed, const void* bias_bf16,
                                             void* out_bf16, mxfp8_stream_t stream) {
  if (B < 1 || M < 0 || N < 1 || K < 1 || K % 32 != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_linear_noalloc: bad B, M, N or K");
  if (K % 128 != 0 || N % 8 != 0)
    return fail(MXFP8_ERR_UNSUPPORTED, "mxfp8_linear_noalloc: needs K % 128 == 0 and N % 8 == 0");
  if (B * M > (1ll << 31) || N > (1ll << 30) || K > (1ll << 30))
    return fail(MXFP8_ERR_UNSUPPORTED, "mxfp8_linear_noalloc: problem too large");
  if (M == 0) return MXFP8_OK;
  if (x_bf16 == nullptr || w_packed == nullptr || sf_packed == nullptr || out_bf16 == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_linear_noalloc: null pointer");
  if (!aligned(x_bf16, 16) || !aligned(w_packed, 16) || !aligned(sf_packed, 16) ||
      !aligned(out_bf16, 16) || (bias_bf16 != nullptr && !aligned(bias_bf16, 16)))
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_linear_noalloc: pointers must be 16-byte aligned");
  uint8_t* scratch = nullptr;
  int sms = 0;
  mxfp8_status st = scratch_for_current_device(&scratch, &sms);
  if (st != MXFP8_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const int dec_splits = (B == 1 && M > 32 && M <= mx::kDecodeMaxM) ? mx::decode_k_splits(M, N, K, sms) : 1;
  if (B == 1 && (M <= 32 || (M <= 64 && dec_splits >= 2) ||
                 (M <= mx::kDecodeMaxM && dec_splits >= 2 && K / dec_splits <= 1024))) {
    // the small-M kernel quantises x inside the GEMM and needs no scratch
    // (the shapes mxfp8_linear's automatic path gives it)
    mx::DecodeProblem p{x_bf16, w_packed, sf_packed, bias_bf16, out_bf16, M, N, K};
    const char* msg = "";
    e = mx::launch_gemm_decode(p, sms, s, &msg);
    if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: small-M GEMM launch failed");
    return MXFP8_OK;
  }
  const int64_t xq_bytes = round_up(B * M * K, 256);
  const int64_t sfa_bytes = round_up(mx::sf_packed_bytes(B, M, K), 256);
  if (xq_bytes + sfa_bytes > kNoallocScratchBytes)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "mxfp8_linear_noalloc: B*M*K plus the packed scales exceeds the fixed scratch "
                "(MXFP8_NOALLOC_SCRATCH_BYTES); use mxfp8_linear with a workspace");
  uint8_t* xq = scratch;
  uint8_t* sfa = scratch + xq_bytes;
  e = mx::launch_quantize(x_bf16, B * M, K, xq, sfa, true, B, M, sms, s, true);
  if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: quantize launch failed");
  mx::GemmProblem p{xq, w_packed, sfa, sf_packed, bias_bf16, out_bf16, B, M, N, K};
  const char* msg = "";
  e = mx::launch_gemm_prefill(p, sms, s, &msg);
  if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "mxfp8_linear_noalloc: GEMM launch failed");
  return MXFP8_OK;
}
