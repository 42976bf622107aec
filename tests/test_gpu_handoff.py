"""The quantised hand-off: a GEMM epilogue that writes its output already
MXFP8-quantised for the next layer (mxfp8_linear_quantized_out,
mxfp8_gemm_packed_quantized_out), the QuantizedActivation path of the
aiter_flydsl page's apply_weights.

* the bf16 output is bit for bit the one mxfp8_linear computes on the same
  kernel;
* the hand-off codes and scales are bit for bit oracle.quantize of that bf16
  output (and the standalone quantiser's bytes);
* a chain of layers fed by the hand-off equals the chain fed by bf16 outputs
  re-quantised (bit for bit, same kernels) and the oracle (tolerance).
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, bf16_bits, bf16_to_dev, device, oracle_weights, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _pack(p, dev):
    wq, ws = oracle_weights(p)
    batched = p.B > 1
    pw = ops.process_weights(u8_to_dev(wq if batched else wq[0], dev), u8_to_dev(ws if batched else ws[0], dev))
    return pw, wq, ws


def _unpacked_scales(pa: ops.PackedActivation) -> np.ndarray:
    """Row-major [B, M, N/32] scales of a hand-off (mxfp8_unpack_scales on its atoms)."""
    out = torch.empty((pa.B, pa.M, pa.K // 32), dtype=torch.uint8, device=pa.x_q.device)
    ops._check(ops.load().mxfp8_unpack_scales(pa.sf_packed.data_ptr(), pa.B, pa.M, pa.K, out.data_ptr(),
                                              ops._stream()))
    return out.cpu().numpy()


def _same_kernel(M, B, N):
    """The kernel gemm_packed and gemm_packed_quantized_out take at these test
    shapes (K <= 512), as a forced path (restated from the library's rule: the
    small-M kernel for B = 1 and M <= 64 -- its K split is at most K / 128 <= 4,
    so the hand-off may use it too; else the unsplit large-M kernels: CTA
    pairs above 128 rows, or while one wave of pairs holds every 256-column
    tile; else one CTA per 128 x 256 tile)."""
    if B == 1 and M <= 64:
        return 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 3 if M > 128 or B * -(-N // 256) * 2 <= sms else 2


# the large-M kernels, split-K included: what the hand-off of a linear call
# runs beyond decode sizes, so its bf16 output must match this path bit for bit
HAND_OFF_PATH = 4


# ref_path: the kernels whose bf16 output the hand-off's must equal -- mxfp8_linear's
# own choice (0); None where its small-M kernel splits K eight ways (8 weight
# tiles, 16 K tiles: 8 clusters of 8 fit) and the hand-off splits four ways:
# there the bf16 output is checked against the oracle within tolerance
@pytest.mark.parametrize("B,M,N,K,bias,ref_path", [(1, 300, 512, 1024, True, 0), (1, 64, 256, 512, False, 0),
                                                   (1, 1, 128, 256, True, 0), (2, 200, 384, 256, True, 0),
                                                   (1, 520, 1024, 384, False, 0), (1, 1, 4096, 4096, True, 0),
                                                   (1, 16, 14336, 4096, True, 0), (1, 100, 4096, 4096, False, 0),
                                                   (1, 16, 1024, 2048, True, None)])
def test_hand_off_bytes_equal_the_oracle_quantiser(B, M, N, K, bias, ref_path):
    dev = device()
    p = synth.make_problem("handoff", B, M, N, K, seed=B * 100 + M + N, bias_std=0.1 if bias else None,
                           x_dist="laplace")
    pw, wq, ws = _pack(p, dev)
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    b = None if p.bias is None else bf16_to_dev(p.bias, dev)
    out, y = ops.linear_quantized_out(x, pw, b)
    if ref_path is None:
        xq64, xs64 = oracle.quantize(synth.bf16_bits_to_f64(p.x[0]))
        assert_close(out, oracle.linear(xq64, xs64, wq[0], ws[0], synth.bf16_bits_to_f64(p.bias)), "hand-off")
    else:
        ref = ops.linear(x, pw, b, path=ref_path)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "bf16 output differs from mxfp8_linear"
    ops.check()

    o64 = synth.bf16_bits_to_f64(bf16_bits(out)).reshape(B, M, N)
    q_ref, s_ref = oracle.quantize(o64)
    assert np.array_equal(y.x_q.cpu().numpy(), q_ref), "hand-off codes differ from oracle.quantize"
    assert np.array_equal(_unpacked_scales(y), s_ref), "hand-off scales differ from oracle.quantize"

    # the standalone quantiser on the bf16 output writes the same bytes
    pa = ops.quantize_packed(out.view(B, M, N), B)
    torch.cuda.synchronize()
    assert torch.equal(pa.x_q, y.x_q)
    assert np.array_equal(_unpacked_scales(pa), _unpacked_scales(y))

    # without the bf16 output the hand-off is unchanged
    none, y2 = ops.linear_quantized_out(x, pw, b, bf16_out=False)
    ops.check()
    assert none is None and torch.equal(y2.x_q, y.x_q)
    assert np.array_equal(_unpacked_scales(y2), s_ref)


def test_hand_off_from_prequantised_input():
    dev = device()
    p = synth.make_problem("handoff-pq", 1, 300, 256, 512, seed=5, bias_std=0.1)
    pw, _, _ = _pack(p, dev)
    xq, xs = ops.quantize(bf16_to_dev(p.x[0], dev))
    b = bf16_to_dev(p.bias, dev)
    out, y = ops.linear_quantized_out(xq, pw, b, x_scale=xs)
    ref = ops.linear(xq, pw, b, x_scale=xs, path=HAND_OFF_PATH)
    ops.check()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    q_ref, s_ref = oracle.quantize(synth.bf16_bits_to_f64(bf16_bits(out))[None])
    assert np.array_equal(y.x_q.cpu().numpy(), q_ref) and np.array_equal(_unpacked_scales(y), s_ref)


@pytest.mark.parametrize("M", [48, 384])
def test_three_layer_chain(M):
    """x -> L1 (hand-off) -> L2 (packed in, hand-off out) -> L3 (packed in, bf16):
    bit for bit the chain of bf16 calls on the same kernels, and within the
    tolerance of the oracle chain (each layer's bf16 output re-quantised)."""
    dev = device()
    dims = [512, 384, 256, 256]        # K of L1, then N of L1..L3
    probs = [synth.make_problem(f"chain{i}", 1, M, dims[i + 1], dims[i], seed=60 + i, bias_std=0.1)
             for i in range(3)]
    layers = [_pack(p, dev) for p in probs]
    biases = [bf16_to_dev(p.bias, dev) for p in probs]
    x = bf16_to_dev(probs[0].x[0], dev)

    _, y1 = ops.linear_quantized_out(x, layers[0][0], biases[0], bf16_out=False)
    _, y2 = ops.gemm_packed_quantized_out(y1, layers[1][0], biases[1], bf16_out=False)
    out3 = ops.gemm_packed(y2, layers[2][0], biases[2])[0]
    ops.check()

    # layer 1 as the hand-off call runs it (mxfp8_linear's choice); layers 2 and 3
    # as gemm_packed and gemm_packed_quantized_out do
    h = x
    for i, ((pw, _, _), b) in enumerate(zip(layers, biases)):
        h = ops.linear(h, pw, b, path=0 if i == 0 else _same_kernel(M, 1, pw.N))
    ops.check()
    assert torch.equal(out3.view(torch.int16), h.view(torch.int16)), "hand-off chain differs from bf16 chain"

    # the oracle chain: each layer's output rounded to bf16 as the layer does, then re-quantised
    h64 = synth.bf16_bits_to_f64(probs[0].x[0])
    for i, (pw, wq, ws) in enumerate(layers):
        xq, xs = oracle.quantize(h64)
        ref = oracle.linear(xq, xs, wq[0], ws[0], synth.bf16_bits_to_f64(probs[i].bias))
        if i < 2:
            h64 = synth.bf16_bits_to_f64(synth.to_bf16_bits(ref))
    assert_close(out3, ref, "three-layer chain")
