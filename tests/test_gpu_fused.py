"""The linear layer with x quantised inside the GEMM (path 5 of mxfp8_linear_path).

The fused kernel reads bf16 x into shared memory and quantises it there, with
the same per-block function as the standalone quantise kernel, into the MMA's
operand tile; its MMA shape (128 x 256 tiles on one CTA) is the one-CTA
GEMM's.  So:
* on integer operands the result equals bf16(oracle) bit for bit;
* on seeded problems it equals the unfused one-CTA path (path 2: standalone
  quantise, then the one-CTA GEMM) bit for bit, and is within the parity
  tolerance of the oracle: ragged M and N, batches, bias, K from one ring
  round to many, MXFP6 weights;
* at the full batched shape (B = 16, M = N = 512, K = 7168) path 5 and path 2
  agree bit for bit on every output of three calls, and sampled batches match
  the oracle;
* inside a CUDA graph, chained calls give the eager results;
* shapes outside its range are refused before any launch.
The exact rounding cases of the quantiser (ties, saturation, subnormals,
zero and clamped blocks) go through this path in test_gpu_rounding.py.
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, bf16_bits, bf16_to_dev, device, oracle_weights, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu

FUSED = 5
UNFUSED_SAME_MMA = 2


def _pack(wq, ws, B, dev, fmt="e4m3"):
    return ops.process_weights(u8_to_dev(wq if B > 1 else wq[0], dev), u8_to_dev(ws if B > 1 else ws[0], dev), fmt)


@pytest.mark.parametrize("B,M,N,K", [(1, 128, 256, 128), (2, 200, 264, 512), (4, 512, 512, 1024),
                                     (1, 1, 8, 256), (3, 130, 136, 384), (1, 77, 512, 4096)])
def test_integer_operands_exact(B, M, N, K):
    """Integer x in [-8, 8] quantises exactly (every block's codes are k * 2^s
    with |k| <= 8) and integer E4M3 weights with unit scales make every fp32
    sum exact: the output must be bf16(oracle) bit for bit."""
    dev = device()
    rng = np.random.default_rng(B * 1000 + M + N + K)
    xi = rng.integers(-8, 9, (B, M, K)).astype(np.float64)
    wi = rng.integers(-8, 9, (B, N, K)).astype(np.float64)
    wq = oracle.e4m3_encode(wi)
    ws = np.full((B, N, K // 32), 127, np.uint8)
    pw = _pack(wq, ws, B, dev)
    x = bf16_to_dev(synth.to_bf16_bits(xi if B > 1 else xi[0]), dev)
    out = ops.linear(x, pw, path=FUSED)
    ops.check()
    exp = synth.to_bf16_bits(np.matmul(xi, np.swapaxes(wi, 1, 2)))
    got = bf16_bits(out).reshape(exp.shape)
    assert np.array_equal(got, exp), f"{int((got != exp).sum())} mismatches"


@pytest.mark.parametrize("B,M,N,K,bias,dist", [(1, 300, 264, 1024, True, "normal"),
                                               (3, 200, 512, 768, False, "laplace"),
                                               (16, 64, 512, 2048, True, "normal"),
                                               (2, 129, 8, 4096, True, "normal"),
                                               (5, 512, 136, 384, True, "laplace")])
def test_equals_unfused_and_oracle(B, M, N, K, bias, dist):
    dev = device()
    p = synth.make_problem("fused", B, M, N, K, seed=B * 7 + M + N, x_dist=dist, bias_std=0.1 if bias else None)
    wq, ws = oracle_weights(p)
    pw = _pack(wq, ws, B, dev)
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    b = None if p.bias is None else bf16_to_dev(p.bias, dev)
    fused = ops.linear(x, pw, b, path=FUSED)
    unfused = ops.linear(x, pw, b, path=UNFUSED_SAME_MMA)
    ops.check()
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16)), \
        "fused quantisation differs from the standalone quantiser on the same MMA shape"
    xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x))
    ref = oracle.linear(xq, xs, wq, ws, None if p.bias is None else synth.bf16_bits_to_f64(p.bias))
    assert_close(fused if B > 1 else fused[None], ref, f"fused B={B} M={M} N={N} K={K}")


def test_batched_workload_matches():
    """B = 16, M = N = 512, K = 7168 (the batched workload): three fused calls
    each equal path 2 bit for bit (a race between the staging ring and the
    quantiser would show as a call that differs), and four batches match the
    oracle."""
    dev = device()
    p = synth.bmm()
    wq, ws = oracle_weights(p)
    pw = _pack(wq, ws, p.B, dev)
    x = bf16_to_dev(p.x, dev)
    unfused = ops.linear(x, pw, path=UNFUSED_SAME_MMA)
    for _ in range(3):
        fused = ops.linear(x, pw, path=FUSED)
        ops.check()
        assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))
    for bi in (0, 5, 10, 15):
        xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x[bi]))
        ref = oracle.linear(xq, xs, wq[bi], ws[bi])
        assert_close(fused[bi], ref, f"batched workload, batch {bi}")


@pytest.mark.parametrize("fmt", ["e2m3", "e3m2"])
def test_mxfp6_weights(fmt):
    dev = device()
    B, M, N, K = 4, 256, 512, 1024
    p = synth.make_problem("fused-fp6", B, M, N, K, seed=55, bias_std=0.1)
    wq, ws = ops.quantize_weights(bf16_to_dev(p.w.reshape(B * N, K), dev), fmt)
    pw = ops.process_weights(wq.view(B, N, K), ws.view(B, N, K // 32), fmt)
    x = bf16_to_dev(p.x, dev)
    b = bf16_to_dev(p.bias, dev)
    fused = ops.linear(x, pw, b, path=FUSED)
    unfused = ops.linear(x, pw, b, path=UNFUSED_SAME_MMA)
    ops.check()
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))
    rq, rs = oracle.quantize_fp6(synth.bf16_bits_to_f64(p.w), fmt)
    xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x))
    ref = oracle.linear(xq, xs, rq, rs, synth.bf16_bits_to_f64(p.bias), w_format=fmt)
    assert_close(fused, ref, f"fused with {fmt} weights")


def test_chained_calls_in_graph_match_eager():
    """Three batched layers (N = K = 512) captured in one CUDA graph with
    path 5: each call's x is the previous call's output, read after the
    kernel's dependency wait."""
    dev = device()
    B, M, N = 8, 512, 512
    g = torch.Generator(device="cpu").manual_seed(3)
    pws = []
    for _ in range(3):
        w = (torch.randn(B, N, N, generator=g) / np.sqrt(N)).to(torch.bfloat16).to(dev)
        wq, ws = ops.quantize(w.view(B * N, N))
        pws.append(ops.process_weights(wq.view(B, N, N), ws.view(B, N, N // 32)))
    bias = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16).to(dev)
    x0 = torch.randn(B, M, N, generator=g).to(torch.bfloat16).to(dev)

    def chain():
        h = x0
        outs = []
        for pw in pws:
            h = ops.linear(h, pw, bias, path=FUSED)
            outs.append(h)
        return outs

    eager = chain()
    torch.cuda.synchronize()
    ops.check()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        outs = chain()
    for o in outs:
        o.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ops.check()
    for i, (e, o) in enumerate(zip(eager, outs)):
        assert torch.equal(e.view(torch.int16), o.view(torch.int16)), f"layer {i} differs from the eager call"


def test_out_of_range_shapes_are_refused():
    dev = device()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    K = 256
    w = torch.zeros((1024, K), dtype=torch.bfloat16, device=dev)
    wq, ws = ops.quantize(w)
    wide = ops.process_weights(wq, ws)                      # N = 1024 > 512
    narrow = ops.process_weights(wq[:512].contiguous(), ws[:512].contiguous())
    x = torch.zeros((128, K), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ops.MxStatusError) as e:
        ops.linear(x, wide, path=FUSED)
    assert e.value.status == 2
    xq, xs = ops.quantize(x)
    with pytest.raises(ops.MxStatusError) as e:             # pre-quantised x: nothing to fuse
        ops.linear(xq, narrow, x_scale=xs, path=FUSED)
    assert e.value.status == 2
    tall = torch.zeros(((sms + 1) * 128 // 2 * 2, K), dtype=torch.bfloat16, device=dev)
    assert -(-tall.shape[0] // 128) * 2 > sms                # more 128 x 256 tiles than SMs
    with pytest.raises(ops.MxStatusError) as e:
        ops.linear(tall, narrow, path=FUSED)
    assert e.value.status == 2
    ops.check()
