"""mxfp8_linear_noalloc: the linear layer for callers that cannot allocate.

Some callers cannot call cudaMalloc at all (their GPU memory is owned by
another pool, or their runtime forbids allocation after start-up), so this
entry point takes no workspace and keeps its scratch in a fixed array inside
the library.  The tests call it through the C ABI (and through the Python
binding with a preallocated output) and check its output against the
workspace-based mxfp8_linear:

* bit for bit against mxfp8_linear_path on the same GEMM kernel (the one-CTA
  kernel up to 128 rows, the CTA-pair kernel above): both run the same
  quantise kernel and the same GEMM, so the bytes must agree;
* within the parity tolerance against mxfp8_linear's own choice (which takes
  the fused small-M kernel up to 64 rows, a different summation order).

Two calls in a row share the scratch array, so the second must not see the
first one's data; a call after the first allocates no device memory.  The
file is collected last, so that a run stopping at the first failure has run
all the other tests before it.
"""

import ctypes
import gc

import numpy as np
import pytest
import torch

import oracle
from _helpers import bf16_to_dev, device, tolerance_violations, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu

N, K = 512, 1024


def _noalloc_abi(x, pw, bias, M):
    """One raw C-ABI call of mxfp8_linear_noalloc (no Python wrapper in between)."""
    out = torch.empty((pw.B, M, pw.N), dtype=torch.bfloat16, device=x.device)
    st = ops.load().mxfp8_linear_noalloc(
        x.data_ptr(), pw.B, M, pw.N, pw.K, pw.w_packed.data_ptr(), pw.sf_packed.data_ptr(),
        None if bias is None else bias.data_ptr(), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, ops.load().mxfp8_last_error().decode()
    return out


def _problem(B, M, seed, x_dist="normal"):
    dev = device()
    p = synth.make_problem(f"noalloc-B{B}-M{M}", B, M, N, K, seed=seed, bias_std=0.1, x_dist=x_dist)
    wq, ws = oracle.quantize(synth.bf16_bits_to_f64(p.w if B > 1 else p.w[0]))
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev))
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    return pw, x, bf16_to_dev(p.bias, dev)


def _same_kernel_path(B, M):
    """The kernel the no-alloc call runs, as a forced path (restated from the
    library's rule: the small-M kernel for B = 1 and M <= 32, or M <= 64
    where it splits K, or M <= 128 where it splits K into ranges of at most
    1024 -- all of these at N = 512, K = 1024: 4 weight tiles, 8 K tiles;
    else CTA pairs above 128 rows, or while one wave of pairs holds every
    256-column tile; else one CTA per 128 x 256 tile)."""
    if B == 1 and M <= 128:
        return 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 3 if M > 128 or B * -(-N // 256) * 2 <= sms else 2


def _assert_close(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64).reshape(-1, got.shape[-1])
    r = ref.float().cpu().numpy().astype(np.float64).reshape(-1, ref.shape[-1])
    bad = tolerance_violations(g, r)
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs outside tolerance"


def test_noalloc_matches_linear_on_two_calls_in_a_row():
    """Two C-ABI calls back to back (different M, inputs and bias) against the
    workspace-based entry point."""
    dev = device()
    pw, x1, bias = _problem(1, 300, seed=31)
    p2 = synth.make_problem("noalloc-2", 1, 1000, N, K, seed=32, x_dist="laplace")
    x2 = bf16_to_dev(p2.x[0], dev)

    a1 = _noalloc_abi(x1, pw, bias, 300)     # two calls in a row share the scratch
    a2 = _noalloc_abi(x2, pw, None, 1000)
    ops.check()
    r1 = ops.linear(x1, pw, bias, path=_same_kernel_path(1, 300))
    r2 = ops.linear(x2, pw, path=_same_kernel_path(1, 1000))
    ops.check()
    assert torch.equal(a1[0].view(torch.int16), r1.view(torch.int16))
    assert torch.equal(a2[0].view(torch.int16), r2.view(torch.int16))
    _assert_close(a1[0], ops.linear(x1, pw, bias), "first call")
    _assert_close(a2[0], ops.linear(x2, pw), "second call")


@pytest.mark.parametrize("B,M", [(1, 1), (1, 64), (1, 128), (1, 300), (3, 96), (2, 300)])
def test_noalloc_binding_equals_linear(B, M):
    """ops.linear_noalloc into a preallocated output, twice, on the one-CTA and
    the CTA-pair kernels and with per-batch packed scales in the scratch."""
    pw, x, bias = _problem(B, M, seed=40 + 7 * B + M)
    out = torch.empty((*x.shape[:-1], N), dtype=torch.bfloat16, device=x.device)
    ops.linear_noalloc(x, pw, bias, out=out)
    same = ops.linear(x, pw, bias, path=_same_kernel_path(B, M))
    ops.check()
    assert torch.equal(out.view(torch.int16), same.view(torch.int16)), \
        "noalloc differs from the workspace path on the same kernels"
    _assert_close(out, ops.linear(x, pw, bias), f"B={B} M={M}")

    # a second call on other data into the same output
    x2 = torch.flip(x, dims=[-2]).contiguous()
    ops.linear_noalloc(x2, pw, None, out=out)
    same2 = ops.linear(x2, pw, None, path=_same_kernel_path(B, M))
    ops.check()
    assert torch.equal(out.view(torch.int16), same2.view(torch.int16))


def test_noalloc_call_allocates_no_device_memory():
    """After the first call on a device (which looks up the scratch address),
    a call changes neither torch's allocator nor the device's free memory."""
    pw, x, bias = _problem(1, 256, seed=77)
    out = torch.empty((256, N), dtype=torch.bfloat16, device=x.device)
    ops.linear_noalloc(x, pw, bias, out=out)
    # free what earlier code left for the garbage collector first, so that
    # the counts below see only the calls
    gc.collect()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        ops.linear_noalloc(x, pw, bias, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0


def test_noalloc_rejects_problems_larger_than_its_scratch():
    dev = device()
    lib = ops.load()
    buf = torch.empty(1 << 12, dtype=torch.uint8, device=dev)
    p = buf.data_ptr()
    # 8192 x 8192 activations need 64 MiB of scratch: refused before any launch
    st = lib.mxfp8_linear_noalloc(p, 1, 8192, 4096, 8192, p, p, None, p,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == 2
    assert b"scratch" in lib.mxfp8_last_error()
    torch.cuda.synchronize()
    assert ctypes.sizeof(ctypes.c_void_p) == 8
