"""Chained linear calls inside a CUDA graph give the eager results bit for bit.

The decode kernel and the CTA-pair GEMM start early under programmatic
dependent launch and wait (griddepcontrol.wait) before they read the previous
kernel's output.  Here each call's input is the previous call's output, so a
read before that wait would change the result; eager calls are the reference
(the kernels are deterministic).
"""

import numpy as np
import pytest
import torch

from _helpers import bf16_bits, device
from mxfp8_block_scaled_02_gb300 import ops

pytestmark = pytest.mark.gpu


def _weights(n_layers, N, K, dev, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    pws = []
    for _ in range(n_layers):
        w = (torch.randn(N, K, generator=g) / np.sqrt(K)).to(torch.bfloat16).to(dev)
        wq, ws = ops.quantize(w)
        pws.append(ops.process_weights(wq, ws))
    bias = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16).to(dev)
    return pws, bias


@pytest.mark.parametrize("M,K", [(1, 1024), (16, 2048), (64, 1024), (512, 1024)])
def test_chained_calls_in_graph_match_eager(M, K):
    dev = device()
    N = K  # each output is the next call's input
    layers = 4
    pws, bias = _weights(layers, N, K, dev, seed=M + K)
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
