"""Calls on two streams at once give the results of the same calls in sequence.

The library keeps no per-call state outside the caller's buffers (each call
gets its own workspace; only mxfp8_linear_noalloc shares a fixed scratch
array, and it documents that overlapping calls race), so interleaving calls
of every kernel path on two streams must not change a single output bit.
The kernels are deterministic, so the sequential results are the reference.
"""

import pytest
import torch

from _helpers import device
from mxfp8_block_scaled_02_gb300 import ops

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, dev, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).to(dev)


def _case(M, N, K, seed, dev, fmt="e4m3"):
    w = _bf16((N, K), seed, dev, 0.05)
    wq, ws = ops.quantize(w) if fmt == "e4m3" else ops.quantize_weights(w, fmt)
    pw = ops.process_weights(wq, ws, fmt)
    x = _bf16((M, K), seed + 1, dev)
    bias = _bf16((N,), seed + 2, dev, 0.1)
    return x, pw, bias


def test_two_streams_match_sequential_calls():
    dev = device()
    cases = [_case(1, 4096, 4096, 1, dev),          # small-M kernel
             _case(300, 1024, 2048, 2, dev),        # CTA pairs
             _case(256, 2048, 4096, 3, dev),        # split-K + reduce
             _case(40, 512, 1024, 4, dev, "e2m3"),  # small-M, MXFP6 weights
             _case(700, 512, 512, 5, dev),          # CTA pairs, two row tiles
             _case(100, 1032, 1024, 6, dev),        # 128-token small-M shape, x quantised once into the workspace
             _case(40, 264, 9216, 7, dev),          # 64-token shape on codes quantised once
             _case(16, 1024, 4096, 8, dev)]         # small-M; its hand-off splits K four ways instead of eight

    def run_all():
        outs = []
        for x, pw, bias in cases:
            outs.append(ops.linear(x, pw, bias))
            if pw.fmt == "e4m3" and pw.N % 128 == 0 and x.shape[0] > 1:
                _, y = ops.linear_quantized_out(x, pw, bias, bf16_out=False)
                outs.append(y.x_q)
        return outs

    ref = run_all()
    torch.cuda.synchronize()
    ops.check()

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    got = []
    for rep in range(3):
        with torch.cuda.stream(s1):
            a = run_all()
        with torch.cuda.stream(s2):
            b = run_all()
        got.append((a, b))
    torch.cuda.synchronize()
    _check_status(s1, s2)
    for a, b in got:
        for i, (r, x1, x2) in enumerate(zip(ref, a, b)):
            assert torch.equal(r.view(torch.uint8), x1.view(torch.uint8)), f"output {i} differs on stream 1"
            assert torch.equal(r.view(torch.uint8), x2.view(torch.uint8)), f"output {i} differs on stream 2"


def _check_status(*streams):
    for s in streams:
        with torch.cuda.stream(s):
            ops.check()
