"""Guard bands around every buffer a library call writes.

compute-sanitizer is not available where these tests run, so out-of-bounds
writes are caught the plain way: each output (and each workspace) is the
middle of a larger device buffer whose 4 KB bands before and after it hold a
canary byte, the call gets exactly the documented number of bytes, and after
the call (and mxfp8_check) both bands must still hold only the canary.  The
calls go through the C ABI with raw pointers, on ragged shapes (M not a
multiple of 128, N not a multiple of 256, batches) and on every kernel path
(small-M, one CTA per tile, CTA pairs, split-K, fused quantise, the hand-off
epilogues, MXFP6 weights, the no-allocation call).  The values the calls
write are checked elsewhere; here only where they write.
"""

import ctypes

import pytest
import torch

from _helpers import device
from mxfp8_block_scaled_02_gb300 import ops

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; keeps the inner pointer 256-byte aligned
CANARY = 0xA5


class Guarded:
    """A device buffer of `nbytes` inside canary bands."""

    def __init__(self, nbytes: int, dev):
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=dev)

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + GUARD

    def inner(self) -> torch.Tensor:
        return self.buf[GUARD:GUARD + self.nbytes]

    def check(self, what: str) -> None:
        torch.cuda.synchronize()
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        bad_head = int((head != CANARY).sum())
        bad_tail = int((tail != CANARY).sum())
        assert bad_head == 0 and bad_tail == 0, \
            f"{what}: {bad_head} bytes before and {bad_tail} bytes after the {self.nbytes}-byte buffer were written"


def _lib():
    return ops.load()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _ok(status):
    assert status == 0, _lib().mxfp8_last_error().decode()


def _sizes(B, R, K, fmt="e4m3"):
    return ops.packed_sizes(B, R, K, fmt)


def _bf16(shape, seed, dev, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).to(dev)


def _weights(B, N, K, dev, fmt="e4m3", seed=1):
    """Packed weights in guarded buffers (mxfp8_quantize_weights then
    mxfp8_process_weights_fmt, both checked for stray writes)."""
    lib = _lib()
    w = _bf16((B * N, K), seed, dev, 0.05)
    q = Guarded(B * N * K, dev)
    s = Guarded(B * N * K // 32, dev)
    _ok(lib.mxfp8_quantize_weights(w.data_ptr(), B * N, K, ops.WFMT[fmt], q.ptr, s.ptr, _stream()))
    wb, sb = _sizes(B, N, K, fmt)
    wp = Guarded(wb, dev)
    sp = Guarded(sb, dev)
    _ok(lib.mxfp8_process_weights_fmt(ops.WFMT[fmt], q.ptr, s.ptr, B, N, K, wp.ptr, sp.ptr, _stream()))
    _ok(lib.mxfp8_check(_stream()))
    for g, what in ((q, "weight codes"), (s, "weight scales"), (wp, "packed weights"), (sp, "packed weight scales")):
        g.check(f"{fmt} B={B} N={N} K={K} {what}")
    return wp, sp


@pytest.mark.parametrize("rows,K", [(1, 32), (130, 96), (257, 4096), (3, 7168)])
def test_quantize_and_repack_calls(rows, K):
    dev = device()
    lib = _lib()
    x = _bf16((rows, K), rows + K, dev)
    q = Guarded(rows * K, dev)
    s = Guarded(rows * K // 32, dev)
    _ok(lib.mxfp8_quantize(x.data_ptr(), rows, K, q.ptr, s.ptr, _stream()))
    B = 1
    sp = Guarded(_sizes(B, rows, K)[1], dev)
    _ok(lib.mxfp8_pack_scales(s.ptr, B, rows, K, sp.ptr, _stream()))
    un = Guarded(rows * K // 32, dev)
    _ok(lib.mxfp8_unpack_scales(sp.ptr, B, rows, K, un.ptr, _stream()))
    xq = Guarded(rows * K, dev)
    xsp = Guarded(_sizes(B, rows, K)[1], dev)
    _ok(lib.mxfp8_quantize_packed(x.data_ptr(), B, rows, K, xq.ptr, xsp.ptr, _stream()))
    _ok(lib.mxfp8_check(_stream()))
    for g, what in ((q, "codes"), (s, "scales"), (sp, "packed scales"), (un, "unpacked scales"),
                    (xq, "packed-path codes"), (xsp, "packed-path scales")):
        g.check(f"rows={rows} K={K} {what}")
    assert torch.equal(un.inner(), s.inner())


@pytest.mark.parametrize("fmt,B,N,K", [("e4m3", 1, 264, 256), ("e4m3", 3, 130, 512),
                                       ("e2m3", 1, 136, 512), ("e3m2", 2, 264, 1024)])
def test_weight_calls(fmt, B, N, K):
    device()
    _weights(B, N, K, device(), fmt, seed=B + N + K)


# (B, M, N, K, path, weight format, pre-quantised x): every kernel path on ragged shapes
LINEAR_CASES = [
    (1, 1, 264, 256, 1, "e4m3", False),      # small-M kernel
    (1, 33, 520, 1024, 1, "e4m3", False),
    (1, 130, 264, 384, 2, "e4m3", False),    # one CTA per 128 x 256 tile
    (1, 100, 264, 512, 2, "e4m3", True),     # ... with the activation-scale repack
    (3, 200, 520, 512, 3, "e4m3", False),    # CTA pairs
    (2, 300, 264, 512, 3, "e4m3", True),     # ... gathering row-major scales
    (1, 256, 1032, 2048, 4, "e4m3", False),  # split-K over pairs + reduce
    (2, 100, 264, 4096, 4, "e4m3", True),
    (1, 300, 4096, 8192, 0, "e4m3", False),  # 32 tiles split two ways (long K)
    (4, 300, 136, 256, 5, "e4m3", False),    # x quantised inside the GEMM
    (1, 5, 10240, 2048, 1, "e4m3", False),   # ... its deep-ring shape (16 K tiles per CTA, no split)
    (1, 5, 264, 512, 1, "e4m3", True),       # small-M kernel copying a pre-quantised x
    (1, 40, 520, 1024, 0, "e4m3", True),
    (1, 40, 264, 9216, 0, "e4m3", False),    # ... x quantised once into the workspace, then copied
    (1, 100, 1032, 1024, 0, "e4m3", False),  # the 128-token shape (x quantised once, copied) ...
    (1, 100, 1032, 1024, 0, "e4m3", True),   # ... and on a pre-quantised x
    (1, 5, 264, 512, 1, "e3m2", False),      # MXFP6 weights on each kind of kernel
    (1, 130, 264, 512, 3, "e2m3", False),
    (2, 256, 264, 512, 5, "e2m3", False),
    (1, 200, 264, 1024, 0, "e4m3", False),   # the automatic choice
]


@pytest.mark.parametrize("B,M,N,K,path,fmt,quantized", LINEAR_CASES)
def test_linear_paths(B, M, N, K, path, fmt, quantized):
    dev = device()
    lib = _lib()
    wp, sp = _weights(B, N, K, dev, fmt, seed=3 * M + N)
    x = _bf16((B, M, K), M + K, dev)
    bias = _bf16((N,), 5, dev, 0.1)
    xq = xs = None
    if quantized:
        xq, xs = ops.quantize(x.reshape(B * M, K))
    n_ws = ctypes.c_size_t()
    _ok(lib.mxfp8_workspace_size(B, M, N, K, int(quantized), ctypes.byref(n_ws)))
    ws = Guarded(n_ws.value, dev)
    out = Guarded(B * M * N * 2, dev)
    _ok(lib.mxfp8_linear_fmt(path, ops.WFMT[fmt], None if quantized else x.data_ptr(),
                             xq.data_ptr() if quantized else None, xs.data_ptr() if quantized else None,
                             B, M, N, K, wp.ptr, sp.ptr, bias.data_ptr(), out.ptr, ws.ptr, ws.nbytes, _stream()))
    _ok(lib.mxfp8_check(_stream()))
    what = f"path {path} {fmt} B={B} M={M} N={N} K={K}"
    out.check(what + " output")
    ws.check(what + " workspace")


@pytest.mark.parametrize("B,M,N,K,bf16_out", [(1, 130, 256, 384, True), (2, 300, 512, 256, False),
                                              (1, 40, 384, 512, True), (1, 256, 1024, 2048, True)])
def test_hand_off_calls(B, M, N, K, bf16_out):
    """mxfp8_linear_quantized_out (one-CTA, pair and split-K epilogues) and
    mxfp8_gemm_packed_quantized_out / mxfp8_gemm_packed on its output."""
    dev = device()
    lib = _lib()
    wp, sp = _weights(B, N, K, dev, seed=N + K)
    w2p, s2p = _weights(B, N, N, dev, seed=N + 7)
    x = _bf16((B, M, K), M, dev)
    n_ws = ctypes.c_size_t()
    _ok(lib.mxfp8_workspace_size(B, M, N, K, 0, ctypes.byref(n_ws)))
    ws = Guarded(n_ws.value, dev)
    out = Guarded(B * M * N * 2, dev) if bf16_out else None
    yq = Guarded(B * M * N, dev)
    ysf = Guarded(_sizes(B, M, N)[1], dev)
    _ok(lib.mxfp8_linear_quantized_out(x.data_ptr(), None, None, B, M, N, K, wp.ptr, sp.ptr, None,
                                       out.ptr if out else None, yq.ptr, ysf.ptr, ws.ptr, ws.nbytes, _stream()))
    # the next layer reads the hand-off: quantised out again, then plain
    out2 = Guarded(B * M * N * 2, dev)
    yq2 = Guarded(B * M * N, dev)
    ysf2 = Guarded(_sizes(B, M, N)[1], dev)
    _ok(lib.mxfp8_gemm_packed_quantized_out(yq.ptr, ysf.ptr, B, M, N, N, w2p.ptr, s2p.ptr, None, out2.ptr,
                                            yq2.ptr, ysf2.ptr, _stream()))
    out3 = Guarded(B * M * N * 2, dev)
    _ok(lib.mxfp8_gemm_packed(yq2.ptr, ysf2.ptr, B, M, N, N, w2p.ptr, s2p.ptr, None, out3.ptr, _stream()))
    _ok(lib.mxfp8_check(_stream()))
    what = f"hand-off B={B} M={M} N={N} K={K}"
    for g, name in ((ws, "workspace"), (out, "bf16 output"), (yq, "codes"), (ysf, "scales"),
                    (out2, "second layer output"), (yq2, "second layer codes"), (ysf2, "second layer scales"),
                    (out3, "third layer output")):
        if g is not None:
            g.check(f"{what} {name}")


@pytest.mark.parametrize("B,M,N,K", [(1, 1, 264, 256), (2, 300, 264, 512), (1, 130, 520, 384)])
def test_noalloc_call(B, M, N, K):
    dev = device()
    lib = _lib()
    wp, sp = _weights(B, N, K, dev, seed=M)
    x = _bf16((B, M, K), K, dev)
    out = Guarded(B * M * N * 2, dev)
    _ok(lib.mxfp8_linear_noalloc(x.data_ptr(), B, M, N, K, wp.ptr, sp.ptr, None, out.ptr, _stream()))
    _ok(lib.mxfp8_check(_stream()))
    out.check(f"noalloc B={B} M={M} N={N} K={K} output")
