"""The small-M path on a pre-quantised x.

"AiterFlyDSLMxfp8LinearKernel.apply_weights" (aiter_flydsl page) takes the
activation either as bf16, quantised inside the layer, or as the
QuantizedActivation pair (E4M3 codes, row-major E8M0 scales [M, K/32]).  On
the small-M kernel the second form is copied into the operand tiles that the
first is quantised into, so the two give the same bytes whenever the codes
are the quantiser's own; on arbitrary codes and scales the result is checked
against the oracle's fp64 product of the dequantised operands.
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, bf16_to_dev, device, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, dev, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).to(dev)


@pytest.mark.parametrize("M,N,K,fmt,bias", [(1, 4096, 4096, "e4m3", True), (5, 264, 512, "e4m3", False),
                                            (16, 4096, 4096, "e4m3", True), (33, 1032, 2048, "e4m3", True),
                                            (64, 4096, 4096, "e4m3", False), (1, 14336, 4096, "e4m3", True),
                                            (7, 264, 1024, "e2m3", True), (16, 520, 512, "e3m2", False),
                                            (100, 1032, 2048, "e4m3", True), (128, 4096, 4096, "e4m3", False)])
def test_same_bytes_as_bf16_input(M, N, K, fmt, bias):
    """x_q, x_scale = quantize(x): the small-M kernel gives bit for bit what it
    gives on x itself, and path 0 routes both forms to kernels that agree."""
    dev = device()
    w = _bf16((N, K), M + N, dev, 0.05)
    wq, ws = ops.quantize(w) if fmt == "e4m3" else ops.quantize_weights(w, fmt)
    pw = ops.process_weights(wq, ws, fmt)
    x = _bf16((M, K), K + M, dev)
    b = _bf16((N,), N, dev, 0.1) if bias else None
    xq, xs = ops.quantize(x)
    y_bf = ops.linear(x, pw, b, path=1)
    y_q = ops.linear(xq, pw, b, x_scale=xs, path=1)
    y_auto_bf = ops.linear(x, pw, b)
    y_auto_q = ops.linear(xq, pw, b, x_scale=xs)
    torch.cuda.synchronize()
    ops.check()
    assert torch.equal(y_bf.view(torch.int16), y_q.view(torch.int16)), "path 1: pre-quantised x differs"
    assert torch.equal(y_auto_bf.view(torch.int16), y_auto_q.view(torch.int16)), "path 0: the two forms differ"


@pytest.mark.parametrize("M,N,K", [(1, 264, 512), (9, 1032, 1024), (64, 264, 256), (16, 4096, 4096),
                                   (128, 264, 1024), (97, 520, 4096)])
def test_arbitrary_codes_match_oracle(M, N, K):
    """Codes and scales that no quantiser produced (every finite E4M3 code,
    scale bytes 112..141) through the small-M copy and through the one-CTA
    large-M kernel, against the oracle's fp64 product."""
    dev = device()
    seed = M * 7 + N + K
    codes = (synth.uniform(seed, 0, M * K) * 256).astype(np.uint8).reshape(M, K)
    codes[(codes & 0x7F) == 0x7F] = 0x3F        # no NaN codes
    scales = (112 + synth.uniform(seed + 1, 0, M * K // 32) * 30).astype(np.uint8).reshape(M, K // 32)
    p = synth.make_problem("prequant", 1, M, N, K, seed=M + N + K, bias_std=0.1)
    wq, ws = oracle.quantize(synth.bf16_bits_to_f64(p.w[0]))
    bias = synth.bf16_bits_to_f64(p.bias)
    ref = oracle.linear(codes, scales, wq, ws, bias)
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev))
    b = bf16_to_dev(p.bias, dev)
    xq, xs = u8_to_dev(codes, dev), u8_to_dev(scales, dev)
    y1 = ops.linear(xq, pw, b, x_scale=xs, path=1)
    y2 = ops.linear(xq, pw, b, x_scale=xs, path=2)
    torch.cuda.synchronize()
    ops.check()
    assert_close(y1, ref, f"small-M, M={M} N={N} K={K}")
    assert_close(y2, ref, f"one-CTA tiles, M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(40, 264, 9216), (64, 1032, 16384), (33, 10240, 1024), (48, 4096, 4096)])
def test_bf16_rows_33_to_64_route(M, N, K):
    """Beyond 32 rows path 0 may quantise x once into the workspace and run the
    small-M kernel on the codes (when its CTAs would each re-quantise a long K
    range): the bytes are those of the fused small-M kernel (path 1)."""
    dev = device()
    w = _bf16((N, K), N + K, dev, 0.05)
    wq, ws = ops.quantize(w)
    pw = ops.process_weights(wq, ws)
    x = _bf16((M, K), M, dev)
    b = _bf16((N,), K, dev, 0.1)
    y0 = ops.linear(x, pw, b)
    y1 = ops.linear(x, pw, b, path=1)
    torch.cuda.synchronize()
    ops.check()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 1032, 2048), (40, 264, 9216), (64, 520, 512),
                                   (100, 1032, 1024), (128, 4096, 4096)])
def test_packed_operands_match_linear(M, N, K):
    """mxfp8_gemm_packed on mxfp8_quantize_packed(x) at decode sizes (the
    small-M kernel reading the scale atoms) gives the bytes mxfp8_linear gives
    on x."""
    dev = device()
    w = _bf16((N, K), N * 3 + K, dev, 0.05)
    wq, ws = ops.quantize(w)
    pw = ops.process_weights(wq, ws)
    x = _bf16((M, K), M + 5, dev)
    b = _bf16((N,), 9, dev, 0.1)
    y_lin = ops.linear(x, pw, b)
    pa = ops.quantize_packed(x)
    y_pk = ops.gemm_packed(pa, pw, b)
    torch.cuda.synchronize()
    ops.check()
    assert torch.equal(y_lin.view(torch.int16), y_pk.reshape(y_lin.shape).view(torch.int16))


def test_copy_route_without_workspace_gives_the_same_bytes():
    """Rows 33..64 of bf16 x on a long K range quantise x once into the
    workspace; given no workspace, the C ABI runs the small-M kernel's own
    quantiser instead: the same bytes."""
    dev = device()
    M, N, K = 40, 264, 9216
    w = _bf16((N, K), 3, dev, 0.05)
    wq, ws = ops.quantize(w)
    pw = ops.process_weights(wq, ws)
    x = _bf16((M, K), 4, dev)
    b = _bf16((N,), 5, dev, 0.1)
    ref = ops.linear(x, pw, b)                       # with the documented workspace
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st = ops.load().mxfp8_linear(x.data_ptr(), None, None, 1, M, N, K, pw.w_packed.data_ptr(),
                                 pw.sf_packed.data_ptr(), b.data_ptr(), out.data_ptr(), None, 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, ops.load().mxfp8_last_error().decode()
    torch.cuda.synchronize()
    ops.check()
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
