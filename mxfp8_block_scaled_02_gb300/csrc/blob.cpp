// blob.cpp - persistable packed weights: the output of mxfp8_process_weights
// as one self-describing byte blob in host memory.
//
// The Mxfp8LinearKernel page has its weights pre-processed once and then
// reused as they are (supports_pre_processed_weights; the weight-cache daemon
// that hands such weights to later processes).  The packed layout depends only
// on (B, N, K) and on this library's layout version, so a process can write
// the blob once and a later one can copy its two payloads back to the device
// and call mxfp8_linear at once, skipping the repack.  A header records the
// format and the layout, so a blob from another library version is refused
// instead of being read with the wrong layout, and two checksums catch a
// truncated or corrupted file.
//
// Byte layout (all integers little-endian; both supported hosts, x86-64 and
// aarch64, are little-endian, and the bytes are written one at a time so the
// code does not depend on that):
//     0  8 bytes  magic "MXFP8PW1"
//     8  u32      format version (1)
//    12  u32      layout id (1: E4M3 codes K-major; 2 / 3: E2M3 / E3M2 codes
//                 packed to 6 bits, 3K/4 bytes per row; in all three the
//                 scales are 128x4 atoms ordered [batch][K tile][row tile], as
//                 mx_layout.cuh describes)
//    16  u32      flags (bit 0: the weights were batched, [B, N, K])
//    20  u32      0
//    24  i64 B, 32 i64 N, 40 i64 K
//    48  u64      w_bytes  (= B * N * K, or 3BNK/4 for packed FP6)
//    56  u64      sf_bytes (= the packed scale bytes of (B, N, K))
//    64  u64      FNV-1a 64 of the payload (w bytes, then sf bytes)
//    72..119      0
//   120  u64      FNV-1a 64 of bytes 0..119
//   128           w payload, then sf payload (both 16-byte aligned offsets)
// Host code only: no CUDA calls, no device memory.
#include <stdint.h>
#include <string.h>

#include "../../include/mxfp8.h"
#include "mx_kernels.h"
#include "mx_layout.cuh"

namespace {

constexpr char kMagic[8] = {'M', 'X', 'F', 'P', '8', 'P', 'W', '1'};
constexpr uint32_t kFormatVersion = 1;
// layout id = weight format + 1 (MXFP8_WFMT_*)
constexpr uint32_t kLayoutE4M3 = 1;
constexpr uint32_t kLayoutLast = 3;
constexpr size_t kHeaderBytes = MXFP8_BLOB_HEADER_BYTES;

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a(uint64_t h, const uint8_t* p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= kFnvPrime;
  }
  return h;
}

void put_u32(uint8_t* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = static_cast<uint8_t>(v >> (8 * i));
}
void put_u64(uint8_t* p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = static_cast<uint8_t>(v >> (8 * i));
}
uint32_t get_u32(const uint8_t* p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= static_cast<uint32_t>(p[i]) << (8 * i);
  return v;
}
uint64_t get_u64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= static_cast<uint64_t>(p[i]) << (8 * i);
  return v;
}

mxfp8_status fail(mxfp8_status st, const char* msg) {
  mx::set_last_error(msg);
  return st;
}

// Payload sizes for (B, N, K) of weight format fmt; false if the shape is
// invalid or too large.
bool payload_sizes(int64_t B, int64_t N, int64_t K, int fmt, uint64_t* w, uint64_t* sf) {
  if (B < 1 || N < 1 || K < 1 || K % 32 != 0 || B > (1ll << 20) || N > (1ll << 31) || K > (1ll << 30))
    return false;
  if (B * N > (1ll << 40) || B * N > (INT64_MAX / K)) return false;
  if (fmt < MXFP8_WFMT_E4M3 || fmt > MXFP8_WFMT_E3M2 || (fmt != MXFP8_WFMT_E4M3 && K % 128 != 0)) return false;
  *w = static_cast<uint64_t>(fmt == MXFP8_WFMT_E4M3 ? B * N * K : B * N * K / 4 * 3);
  *sf = static_cast<uint64_t>(mx::sf_packed_bytes(B, N, K));
  return true;
}

}  // namespace

extern "C" {

mxfp8_status mxfp8_blob_size(int64_t B, int64_t N, int64_t K, int w_format, size_t* bytes) {
  uint64_t w = 0, sf = 0;
  if (bytes == nullptr) return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_blob_size: null output pointer");
  if (!payload_sizes(B, N, K, w_format, &w, &sf))
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_blob_size: bad B, N, K or w_format");
  *bytes = kHeaderBytes + w + sf;
  return MXFP8_OK;
}

mxfp8_status mxfp8_weights_serialize(const uint8_t* w_packed, const uint8_t* sf_packed, int64_t B,
                                     int64_t N, int64_t K, int w_format, int batched, uint8_t* blob,
                                     size_t blob_bytes) {
  uint64_t w = 0, sf = 0;
  if (w_packed == nullptr || sf_packed == nullptr || blob == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_serialize: null pointer");
  if (!payload_sizes(B, N, K, w_format, &w, &sf))
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_serialize: bad B, N, K or w_format");
  if (blob_bytes < kHeaderBytes + w + sf)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_serialize: blob smaller than mxfp8_blob_size()");
  if (batched != 0 && batched != 1) return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_serialize: batched is 0 or 1");
  uint8_t* h = blob;
  memset(h, 0, kHeaderBytes);
  memcpy(h, kMagic, 8);
  put_u32(h + 8, kFormatVersion);
  put_u32(h + 12, kLayoutE4M3 + static_cast<uint32_t>(w_format));
  put_u32(h + 16, static_cast<uint32_t>(batched));
  put_u64(h + 24, static_cast<uint64_t>(B));
  put_u64(h + 32, static_cast<uint64_t>(N));
  put_u64(h + 40, static_cast<uint64_t>(K));
  put_u64(h + 48, w);
  put_u64(h + 56, sf);
  memcpy(blob + kHeaderBytes, w_packed, w);
  memcpy(blob + kHeaderBytes + w, sf_packed, sf);
  put_u64(h + 64, fnv1a(kFnvOffset, blob + kHeaderBytes, w + sf));
  put_u64(h + 120, fnv1a(kFnvOffset, h, 120));
  return MXFP8_OK;
}

mxfp8_status mxfp8_weights_deserialize(const uint8_t* blob, size_t blob_bytes, int64_t* B, int64_t* N,
                                       int64_t* K, int* w_format, int* batched, size_t* w_offset,
                                       size_t* sf_offset) {
  if (blob == nullptr || B == nullptr || N == nullptr || K == nullptr || w_format == nullptr || batched == nullptr ||
      w_offset == nullptr || sf_offset == nullptr)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: null pointer");
  if (blob_bytes < kHeaderBytes)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: shorter than the header");
  const uint8_t* h = blob;
  if (memcmp(h, kMagic, 8) != 0)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: not a packed-weights blob (magic)");
  if (get_u64(h + 120) != fnv1a(kFnvOffset, h, 120))
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: header checksum mismatch (corrupted)");
  const uint32_t layout = get_u32(h + 12);
  if (get_u32(h + 8) != kFormatVersion || layout < kLayoutE4M3 || layout > kLayoutLast)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "mxfp8_weights_deserialize: blob written with another format version or layout; "
                "repack the weights with mxfp8_process_weights");
  const uint32_t flags = get_u32(h + 16);
  if ((flags & ~1u) != 0 || get_u32(h + 20) != 0)
    return fail(MXFP8_ERR_UNSUPPORTED, "mxfp8_weights_deserialize: unknown header flags");
  const int64_t b = static_cast<int64_t>(get_u64(h + 24));
  const int64_t n = static_cast<int64_t>(get_u64(h + 32));
  const int64_t k = static_cast<int64_t>(get_u64(h + 40));
  const int fmt = static_cast<int>(layout - kLayoutE4M3);
  uint64_t w = 0, sf = 0;
  if (!payload_sizes(b, n, k, fmt, &w, &sf) || get_u64(h + 48) != w || get_u64(h + 56) != sf)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: sizes do not match (B, N, K)");
  if (blob_bytes < kHeaderBytes + w + sf)
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: blob truncated");
  if (get_u64(h + 64) != fnv1a(kFnvOffset, blob + kHeaderBytes, w + sf))
    return fail(MXFP8_ERR_INVALID_ARG, "mxfp8_weights_deserialize: payload checksum mismatch (corrupted)");
  *B = b;
  *N = n;
  *K = k;
  *w_format = fmt;
  *batched = static_cast<int>(flags & 1u);
  *w_offset = kHeaderBytes;
  *sf_offset = kHeaderBytes + w;
  return MXFP8_OK;
}

}  // extern "C"
