"""Chained linear calls inside a CUDA graph give the eager results bit for bit.

The decode kernel and the CTA-pair GEMM start early under programmatic
dependent launch and wait (griddepcontrol.wait) before they read the previous
kernel's output.  Here each call's input is the previous call's output, so a
read before that wait would change the result; eager calls are the reference
(the kernels are deterministic).  Covered: the decode kernel (M <= 64), the
CTA-pair GEMM with and without split-K (whose reduce kernel is a third launch
per call), the quantised hand-off chain, and MXFP6 weights.
"""

import numpy as np
import pytest
import torch

from _helpers import bf16_bits, device
from mxfp8_block_scaled_02_gb300 import ops

pytestmark = pytest.mark.gpu


def _weights(n_layers, N, K, dev, seed, fmt="e4m3"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    pws = []
    for _ in range(n_layers):
        w = (torch.randn(N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16).to(dev)
        wq, ws = ops.quantize(w) if fmt == "e4m3" else ops.quantize_weights(w, fmt)
        pws.append(ops.process_weights(wq, ws, fmt))
    bias = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16).to(dev)
    return pws, bias


def _unpacked_scales(pa):
    """Row-major [B, M, N/32] scales of a hand-off (mxfp8_unpack_scales on its atoms)."""
    out = torch.empty((pa.B, pa.M, pa.K // 32), dtype=torch.uint8, device=pa.x_q.device)
    ops._check(ops.load().mxfp8_unpack_scales(pa.sf_packed.data_ptr(), pa.B, pa.M, pa.K, out.data_ptr(),
                                              ops._stream()))
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _splits(M, N, K):
    """The split count the library picks for one batch (restated from its rule)."""
    tiles = -(-M // 256) * -(-N // 256)
    if tiles > (32 if K // 128 >= 64 else 16):
        return 1
    s = min(64 // tiles, (K // 128) // 4, 8)
    return s if s >= 2 else 1


def _capture(fn, side):
    """Warm fn up on the side stream, then capture it into a graph."""
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        res = fn()
    return graph, res


@pytest.mark.parametrize("M,K,fmt", [(1, 1024, "e4m3"), (16, 2048, "e4m3"), (64, 1024, "e4m3"),
                                     (512, 1024, "e4m3"), (256, 4096, "e4m3"), (1024, 2048, "e4m3"),
                                     (1, 2048, "e2m3"), (512, 1024, "e3m2")])
def test_chained_calls_in_graph_match_eager(M, K, fmt):
    dev = device()
    N = K  # each output is the next call's input
    layers = 4
    if (M, K) == (256, 4096):
        assert _splits(M, N, K) == 4        # four pairs per tile, then the reduce kernel
    if (M, K) == (1024, 2048):
        assert _splits(M, N, K) == 1        # 32 tiles: no split
    pws, bias = _weights(layers, N, K, dev, seed=M + K, fmt=fmt)
    g = torch.Generator(device="cpu").manual_seed(7)
    x0 = torch.randn(M, K, generator=g).to(torch.bfloat16).to(dev)

    eager = []
    x = x0
    for pw in pws:
        x = ops.linear(x, pw, bias)
        eager.append(x)
    torch.cuda.synchronize()
    ops.check()

    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(layers)]
    wss = [torch.empty(max(ops.workspace_size(1, M, N, K, False), 1), dtype=torch.uint8, device=dev)
           for _ in range(layers)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm up on the capture stream
        x = x0
        for pw, o, w in zip(pws, outs, wss):
            x = ops.linear(x, pw, bias, out=o, workspace=w)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        x = x0
        for pw, o, w in zip(pws, outs, wss):
            x = ops.linear(x, pw, bias, out=o, workspace=w)
    for o in outs:
        o.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ops.check()
    for i, (e, o) in enumerate(zip(eager, outs)):
        assert np.array_equal(bf16_bits(e), bf16_bits(o)), f"layer {i} differs from the eager call"


@pytest.mark.parametrize("M", [16, 256, 1024])
def test_hand_off_chain_in_graph_matches_eager(M):
    """linear_quantized_out -> gemm_packed_quantized_out -> gemm_packed captured
    in one graph: each GEMM reads the codes and packed scales its predecessor's
    epilogue wrote."""
    dev = device()
    N = K = 1024
    pws, bias = _weights(3, N, K, dev, seed=90 + M)
    g = torch.Generator(device="cpu").manual_seed(9)
    x0 = torch.randn(M, K, generator=g).to(torch.bfloat16).to(dev)

    def chain():
        o1, y1 = ops.linear_quantized_out(x0, pws[0], bias)
        o2, y2 = ops.gemm_packed_quantized_out(y1, pws[1], bias)
        o3 = ops.gemm_packed(y2, pws[2], bias)
        return o1, o2, o3, y2

    eager = chain()
    torch.cuda.synchronize()
    ops.check()
    graph, outs = _capture(chain, torch.cuda.Stream())
    for t in outs[:3]:
        t.zero_()
    outs[3].x_q.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ops.check()
    for i in range(3):
        assert np.array_equal(bf16_bits(eager[i]), bf16_bits(outs[i])), f"layer {i} differs from the eager call"
    # the codes and the scales of the M real rows (atom padding rows are not
    # written by the hand-off and hold whatever the buffer held)
    assert torch.equal(eager[3].x_q, outs[3].x_q)
    assert np.array_equal(_unpacked_scales(eager[3]), _unpacked_scales(outs[3]))
