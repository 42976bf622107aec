"""Persistable packed weights on CPU: the blob written by
mxfp8_weights_serialize reads back bit for bit, its header has the documented
byte layout (restated here with struct and an FNV-1a written from its
definition), and a corrupted, truncated or foreign blob is refused."""

import ctypes
import struct

import numpy as np
import pytest
import torch

from mxfp8_block_scaled_02_gb300 import build, ops

HEADER = 128


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load()


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: offset basis 0xcbf29ce484222325, prime 0x100000001b3."""
    h = 0xCBF29CE484222325
    for b in data:
        h = ((h ^ b) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _random_packed(B, N, K, batched, seed, fmt="e4m3"):
    rng = np.random.default_rng(seed)
    wb, sb = ops.packed_sizes(B, N, K, fmt)
    w = torch.from_numpy(rng.integers(0, 256, wb, dtype=np.uint8))
    sf = torch.from_numpy(rng.integers(0, 256, sb, dtype=np.uint8))
    return ops.PackedWeights(w, sf, B, N, K, batched, fmt)


@pytest.mark.parametrize("B,N,K,batched,fmt", [(1, 8, 32, False, "e4m3"), (1, 136, 256, False, "e4m3"),
                                               (3, 40, 160, True, "e4m3"), (1, 16, 128, True, "e4m3"),
                                               (1, 24, 256, False, "e2m3"), (2, 8, 128, True, "e3m2")])
def test_round_trip_and_header_layout(lib, B, N, K, batched, fmt):
    pw = _random_packed(B, N, K, batched, seed=B * 1000 + N + K, fmt=fmt)
    blob = ops.save_packed(pw)
    wb, sb = ops.packed_sizes(B, N, K, fmt)
    assert len(blob) == HEADER + wb + sb

    magic, ver, layout, flags, zero, b, n, k, w_bytes, sf_bytes, psum = struct.unpack_from(
        "<8sIIIIqqqQQQ", blob, 0)
    assert magic == b"MXFP8PW1" and ver == 1 and layout == 1 + ops.WFMT[fmt] and zero == 0
    assert flags == int(batched) and (b, n, k) == (B, N, K) and (w_bytes, sf_bytes) == (wb, sb)
    assert blob[72:120] == bytes(48)
    assert psum == fnv1a64(blob[HEADER:])
    assert struct.unpack_from("<Q", blob, 120)[0] == fnv1a64(blob[:120])
    assert blob[HEADER:HEADER + wb] == pw.w_packed.numpy().tobytes()
    assert blob[HEADER + wb:] == pw.sf_packed.numpy().tobytes()

    back = ops.load_packed(blob, "cpu")
    assert (back.B, back.N, back.K, back.batched, back.fmt) == (B, N, K, batched, fmt)
    assert torch.equal(back.w_packed, pw.w_packed) and torch.equal(back.sf_packed, pw.sf_packed)


def _deserialize(lib, blob):
    buf = np.frombuffer(bytes(blob), dtype=np.uint8)
    out = [ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int(), ctypes.c_int(),
           ctypes.c_size_t(), ctypes.c_size_t()]
    st = lib.mxfp8_weights_deserialize(buf.ctypes.data, buf.size, *[ctypes.byref(o) for o in out])
    return st, [o.value for o in out]


def test_corrupted_truncated_and_foreign_blobs_are_refused(lib):
    pw = _random_packed(2, 24, 128, True, seed=5)
    blob = bytearray(ops.save_packed(pw))
    st, vals = _deserialize(lib, blob)
    assert st == 0 and vals[:5] == [2, 24, 128, 0, 1] and vals[5] == HEADER

    bad = bytearray(blob)
    bad[HEADER + 17] ^= 0x01                      # one payload bit
    st, _ = _deserialize(lib, bad)
    assert st == 1 and b"payload checksum" in lib.mxfp8_last_error()

    bad = bytearray(blob)
    struct.pack_into("<q", bad, 32, 25)           # N changed, header checksum stale
    st, _ = _deserialize(lib, bad)
    assert st == 1 and b"header checksum" in lib.mxfp8_last_error()

    bad = bytearray(blob)
    struct.pack_into("<I", bad, 8, 2)             # another format version, consistent checksum
    struct.pack_into("<Q", bad, 120, fnv1a64(bytes(bad[:120])))
    st, _ = _deserialize(lib, bad)
    assert st == 2 and b"format version" in lib.mxfp8_last_error()

    bad = bytearray(blob)
    struct.pack_into("<I", bad, 12, 7)            # another layout
    struct.pack_into("<Q", bad, 120, fnv1a64(bytes(bad[:120])))
    assert _deserialize(lib, bad)[0] == 2

    bad = bytearray(blob)
    struct.pack_into("<Q", bad, 48, 1)            # sizes inconsistent with (B, N, K)
    struct.pack_into("<Q", bad, 120, fnv1a64(bytes(bad[:120])))
    st, _ = _deserialize(lib, bad)
    assert st == 1 and b"sizes" in lib.mxfp8_last_error()

    assert _deserialize(lib, blob[:-1])[0] == 1   # truncated payload
    assert _deserialize(lib, blob[:100])[0] == 1  # truncated header
    bad = bytearray(blob)
    bad[0:8] = b"NOTABLOB"
    st, _ = _deserialize(lib, bad)
    assert st == 1 and b"magic" in lib.mxfp8_last_error()
    with pytest.raises(ops.MxStatusError):
        ops.load_packed(bytes(bad), "cpu")


def test_serialize_argument_errors(lib):
    n = ctypes.c_size_t()
    assert lib.mxfp8_blob_size(1, 8, 48, 0, ctypes.byref(n)) == 1   # K % 32
    assert lib.mxfp8_blob_size(1, 8, 64, 1, ctypes.byref(n)) == 1   # packed FP6 needs K % 128
    assert lib.mxfp8_blob_size(1, 8, 64, 3, ctypes.byref(n)) == 1   # no such weight format
    assert lib.mxfp8_blob_size(1, 8, 128, 2, ctypes.byref(n)) == 0 and n.value == HEADER + 8 * 96 + 512
    assert lib.mxfp8_blob_size(1, 8, 64, 0, ctypes.byref(n)) == 0 and n.value == HEADER + 8 * 64 + 512
    buf = np.zeros(n.value - 1, np.uint8)
    src = np.zeros(4096, np.uint8)
    assert lib.mxfp8_weights_serialize(src.ctypes.data, src.ctypes.data, 1, 8, 64, 0, 0, buf.ctypes.data,
                                       buf.size) == 1             # blob one byte short
    assert lib.mxfp8_weights_serialize(None, src.ctypes.data, 1, 8, 64, 0, 0, buf.ctypes.data,
                                       buf.size + 1) == 1
