"""The C ABI without a GPU: the library builds, loads, exports every declared
symbol, and rejects bad arguments before touching a device."""

import ctypes
import os
import re
import subprocess

import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

from mxfp8_block_scaled_02_gb300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp8.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp8_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["mxfp8_quantize", "mxfp8_process_weights", "mxfp8_linear",
                     "mxfp8_packed_sizes", "mxfp8_workspace_size", "mxfp8_last_error",
                     "mxfp8_check"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ops.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(mxfp8_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    # the binding covers exactly the declared calls
    assert set(ops.SIGNATURES) == set(declared_functions())


def test_version_and_sizes(lib):
    assert lib.mxfp8_version() == 1
    assert ops.packed_sizes(1, 256, 512) == (256 * 512, 2 * 4 * 512)
    assert ops.packed_sizes(16, 512, 7168) == (16 * 512 * 7168, 16 * 56 * 4 * 512)
    # ragged rows and K round up to whole atoms
    assert ops.packed_sizes(1, 129, 160) == (129 * 160, 2 * 2 * 512)
    assert ops.workspace_size(1, 4096, 14336, 4096, False) == 4096 * 4096 + 32 * 32 * 512
    assert ops.workspace_size(1, 8192, 4096, 14336, True) == 64 * 112 * 512


def _status(fn, *args):
    return fn(*args)


def test_argument_errors_are_reported_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails its checks first
    # neither or both activation forms
    st = lib.mxfp8_linear(None, None, None, 1, 16, 256, 512, fake, fake, None, fake, fake, 1 << 20, None)
    assert st == 1 and b"exactly one" in lib.mxfp8_last_error()
    st = lib.mxfp8_linear(fake, fake, fake, 1, 16, 256, 512, fake, fake, None, fake, fake, 1 << 20, None)
    assert st == 1
    # K not a multiple of 32 -> invalid; of 128 -> unsupported
    assert lib.mxfp8_linear(fake, None, None, 1, 16, 256, 500, fake, fake, None, fake, fake, 1 << 20, None) == 1
    assert lib.mxfp8_linear(fake, None, None, 1, 16, 256, 544, fake, fake, None, fake, fake, 1 << 20, None) == 2
    # N not a multiple of 8
    assert lib.mxfp8_linear(fake, None, None, 1, 16, 250, 512, fake, fake, None, fake, fake, 1 << 20, None) == 2
    # misaligned output
    assert lib.mxfp8_linear(fake, None, None, 1, 16, 256, 512, fake, fake, None, P(0x10002), fake,
                            1 << 20, None) == 1
    # bad path selector (0..5 are the paths)
    for bad_path in (-1, 6, 7):
        assert lib.mxfp8_linear_path(bad_path, fake, None, None, 1, 16, 256, 512, fake, fake, None, fake,
                                     fake, 1 << 20, None) == 1
    # quantize: K % 32
    assert lib.mxfp8_quantize(fake, 4, 33, fake, fake, None) == 1
    assert lib.mxfp8_quantize(None, 4, 64, fake, fake, None) == 1
    # process_weights: null scale
    assert lib.mxfp8_process_weights(fake, None, 1, 8, 64, fake, fake, None) == 1
    # sizes: bad K
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.mxfp8_packed_sizes(1, 8, 48, ctypes.byref(a), ctypes.byref(b)) == 1
    assert lib.mxfp8_debug_expire_wait(10, None) == 1


def test_misaligned_scale_pointers_are_refused_before_launch(lib):
    """Every scale pointer is checked like the other tensor pointers: an odd
    address gets MXFP8_ERR_INVALID_ARG before any launch (no GPU here, so a call
    that reached a kernel or a device query would return another status)."""
    P = ctypes.c_void_p
    fake, odd, odd4 = P(0x10000), P(0x10001), P(0x10004)
    # pre-quantised activation scales
    for bad in (odd, odd4):
        assert lib.mxfp8_linear(None, fake, bad, 1, 300, 256, 512, fake, fake, None, fake, fake,
                                1 << 20, None) == 1
        assert b"aligned" in lib.mxfp8_last_error()
        assert lib.mxfp8_linear_path(3, None, fake, bad, 1, 300, 256, 512, fake, fake, None, fake,
                                     fake, 1 << 20, None) == 1
    # weight scales (and the weights) given to the one-time repack
    assert lib.mxfp8_process_weights(fake, odd4, 1, 8, 128, fake, fake, None) == 1
    assert lib.mxfp8_process_weights(odd, fake, 1, 8, 128, fake, fake, None) == 1
    assert lib.mxfp8_process_weights(fake, fake, 1, 8, 128, fake, odd, None) == 1
    # the standalone scale repack, both sides, and its inverse
    assert lib.mxfp8_pack_scales(odd4, 1, 8, 128, fake, None) == 1
    assert lib.mxfp8_pack_scales(fake, 1, 8, 128, odd, None) == 1
    assert lib.mxfp8_unpack_scales(fake, 1, 8, 128, odd, None) == 1
    # row-major activation scales written by the standalone quantiser
    assert lib.mxfp8_quantize(fake, 4, 64, fake, odd, None) == 1
    assert lib.mxfp8_quantize_packed(fake, 1, 4, 64, fake, odd4, None) == 1
    # bias and the no-allocation entry point
    assert lib.mxfp8_linear(fake, None, None, 1, 16, 256, 512, fake, fake, odd, fake, fake,
                            1 << 20, None) == 1
    assert lib.mxfp8_linear_noalloc(fake, 1, 16, 256, 512, fake, odd4, None, fake, None) == 1


def test_quantized_out_argument_errors(lib):
    """The hand-off calls refuse what they cannot do before any launch."""
    P = ctypes.c_void_p
    fake, odd = P(0x10000), P(0x10008)
    # N % 128 != 0: the hand-off feeds a layer with K = N
    assert lib.mxfp8_linear_quantized_out(fake, None, None, 1, 300, 136, 512, fake, fake, None, fake, fake, fake,
                                          fake, 1 << 20, None) == 2
    assert b"N %" in lib.mxfp8_last_error() or b"128" in lib.mxfp8_last_error()
    # both hand-off buffers are required; the bf16 output is optional
    assert lib.mxfp8_linear_quantized_out(fake, None, None, 1, 300, 256, 512, fake, fake, None, fake, None, fake,
                                          fake, 1 << 20, None) == 1
    assert lib.mxfp8_gemm_packed_quantized_out(fake, fake, 1, 300, 256, 512, fake, fake, None, None, fake, None,
                                               None) == 1
    # misaligned hand-off scale buffer
    assert lib.mxfp8_linear_quantized_out(fake, None, None, 1, 300, 256, 512, fake, fake, None, None, fake, odd,
                                          fake, 1 << 20, None) == 1
    assert lib.mxfp8_gemm_packed_quantized_out(fake, fake, 1, 300, 256, 512, fake, fake, None, None, odd, fake,
                                               None) == 1
    # M = 0 is a no-op whatever the pointers
    assert lib.mxfp8_linear_quantized_out(None, None, None, 1, 0, 256, 512, None, None, None, None, None, None,
                                          None, 0, None) == 0


def test_problems_beyond_32_bit_block_indexing_are_unsupported(lib):
    """The quantise and repack kernels index scale blocks with 32-bit integers:
    more than 2^31 - 1 blocks is refused with MXFP8_ERR_UNSUPPORTED up front."""
    fake = ctypes.c_void_p(0x10000)
    rows, K = 1 << 22, 1 << 14            # 2^22 * 2^9 = 2^31 blocks
    assert lib.mxfp8_quantize(fake, rows, K, fake, fake, None) == 2
    assert b"2^31" in lib.mxfp8_last_error()
    assert lib.mxfp8_quantize_packed(fake, 1, rows, K, fake, fake, None) == 2
    assert lib.mxfp8_linear(fake, None, None, 1, rows, 256, K, fake, fake, None, fake, fake,
                            1 << 62, None) == 2
    assert lib.mxfp8_process_weights(fake, fake, 1, rows, K, fake, fake, None) == 2
    assert lib.mxfp8_pack_scales(fake, 2, rows // 2, K, fake, None) == 2
    # one block fewer than the limit is accepted by the size checks (the call
    # then fails on the missing GPU, not on its arguments)
    st = lib.mxfp8_quantize(fake, rows - 1, K, fake, fake, None)
    assert st not in (1, 2)


def test_python_binding_validates_shapes():
    with pytest.raises(TypeError):
        ops.quantize(torch.zeros(4, 64, dtype=torch.float32))
    with pytest.raises(ValueError):
        ops.quantize(torch.zeros(4, 64, dtype=torch.bfloat16))   # CPU tensor


def test_build_entry_point_is_importable():
    import __graft_entry__ as g
    assert callable(g.build) and callable(g.smoke)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    # no fallback path: without the built library every call raises
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="is missing"):
        ops.load(str(tmp_path / "libmxfp8.so"))


def test_workspace_size_follows_the_split_rule(lib):
    """mxfp8_workspace_size (host only) includes 4 * splits * B * M * N bytes
    of split-K partials exactly when the shape is split: at most 16 tiles of
    256 x 256 (at most 32 when K has at least 64 K tiles), min(64 / tiles,
    K tiles / 4, 8) ways, at least 2."""

    def ws(B, M, N, K, quantized=0):
        n = ctypes.c_size_t()
        assert lib.mxfp8_workspace_size(B, M, N, K, quantized, ctypes.byref(n)) == 0
        return n.value

    def base(B, M, K):
        a, b = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.mxfp8_packed_sizes(B, M, K, ctypes.byref(a), ctypes.byref(b)) == 0
        return -(-(B * M * K) // 256) * 256 + -(-b.value // 256) * 256

    for (B, M, N, K, splits) in [(1, 256, 4096, 4096, 4), (1, 128, 1024, 2048, 4), (1, 512, 4096, 4096, 1),
                                 (1, 512, 4096, 14336, 2), (1, 300, 4096, 8192, 2), (1, 1024, 4096, 14336, 1),
                                 (2, 100, 256, 4096, 8), (1, 4096, 14336, 4096, 1)]:
        parts = 4 * splits * B * M * N if splits > 1 else 0
        assert ws(B, M, N, K) == base(B, M, K) + parts, (B, M, N, K, splits)
