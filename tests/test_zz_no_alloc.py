"""mxfp8_linear_noalloc: the linear layer for callers that cannot allocate.

Some callers cannot call cudaMalloc at all (their GPU memory is owned by
another pool, or their runtime forbids allocation after start-up), so this
entry point takes no workspace and keeps its scratch in a fixed array inside
the library.  The test calls it through the C ABI twice in a row, on
different inputs, and checks each output against the workspace-based
mxfp8_linear with the same tolerance as the other parity tests.  It is
collected last so that a run stopping at the first failure has run all the
other tests before it.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from _helpers import bf16_to_dev, device, tolerance_violations, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _noalloc(x, pw, bias, M):
    out = torch.empty((M, pw.N), dtype=torch.bfloat16, device=x.device)
    st = ops.load().mxfp8_linear_noalloc(
        x.data_ptr(), pw.B, M, pw.N, pw.K, pw.w_packed.data_ptr(), pw.sf_packed.data_ptr(),
        None if bias is None else bias.data_ptr(), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, ops.load().mxfp8_last_error().decode()
    return out


def test_noalloc_matches_linear_on_two_calls_in_a_row():
    dev = device()
    p1 = synth.make_problem("na1", 1, 300, 512, 1024, seed=31, bias_std=0.1)
    p2 = synth.make_problem("na2", 1, 1000, 512, 1024, seed=32, x_dist="laplace")
    wq, ws = oracle.quantize(synth.bf16_bits_to_f64(p1.w[0]))
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev))
    bias = bf16_to_dev(p1.bias, dev)
    x1 = bf16_to_dev(p1.x[0], dev)
    x2 = bf16_to_dev(p2.x[0], dev)

    a1 = _noalloc(x1, pw, bias, p1.M)      # two calls in a row share the scratch
    a2 = _noalloc(x2, pw, None, p2.M)
    ops.check()
    r1 = ops.linear(x1, pw, bias)
    r2 = ops.linear(x2, pw)
    ops.check()
    torch.cuda.synchronize()

    for got, ref in ((a1, r1), (a2, r2)):
        g = got.float().cpu().numpy().astype(np.float64)
        r = ref.float().cpu().numpy().astype(np.float64)
        bad = tolerance_violations(g, r)
        assert not bad.any(), f"{int(bad.sum())} outputs differ from mxfp8_linear"


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
