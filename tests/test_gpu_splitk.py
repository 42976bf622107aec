"""Split-K on CTA pairs for shapes with few output tiles (path 0 / path 4 of
mxfp8_linear_path): each 256 x 256 tile's K range is split over several
pairs, fp32 partials go to the workspace and a reduce kernel adds them in a
fixed order with the bias.

* integer operands: the fp32 partial sums are exact, so the result must equal
  bf16(oracle) bit for bit whatever the split;
* seeded problems: within the parity tolerance of the oracle (and of the
  unsplit CTA-pair path), bias, batches, pre-quantised and MXFP6 weights;
* the same output on every call (fixed summation order);
* the hand-off written by the reduce equals oracle.quantize(bf16 output).
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, bf16_bits, bf16_to_dev, device, oracle_weights, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def splits_for(B, M, N, K):
    """The split count the library uses (restated from its rule)."""
    tiles = B * -(-M // 256) * -(-N // 256)
    if tiles > (32 if K // 128 >= 64 else 16):
        return 1
    s = min(64 // tiles, (K // 128) // 4, 8)
    return s if s >= 2 else 1


def test_workspace_includes_the_partials():
    device()
    B, M, N, K = 1, 256, 4096, 4096
    assert splits_for(B, M, N, K) == 4
    base = -(-(B * M * K) // 256) * 256 + -(-ops.packed_sizes(B, M, K)[1] // 256) * 256
    assert ops.workspace_size(B, M, N, K, False) == base + 4 * B * M * N * 4
    assert splits_for(1, 512, 4096, 4096) == 1                      # 32 tiles: not split
    assert splits_for(1, 512, 4096, 14336) == 2                     # ... unless K is long
    base = -(-(512 * 14336) // 256) * 256 + -(-ops.packed_sizes(1, 512, 14336)[1] // 256) * 256
    assert ops.workspace_size(1, 512, 4096, 14336, False) == base + 2 * 512 * 4096 * 4
    assert ops.workspace_size(1, 4096, 14336, 4096, False) == 4096 * 4096 + 32 * 32 * 512   # no split


@pytest.mark.parametrize("B,M,N,K", [(1, 256, 4096, 4096), (1, 128, 1024, 2048), (1, 300, 520, 1024),
                                     (2, 100, 256, 4096), (1, 1, 256, 1024)])
def test_integer_operands_exact(B, M, N, K):
    dev = device()
    assert splits_for(B, M, N, K) > 1
    rng = np.random.default_rng(M + N + K + B)
    xi = rng.integers(-8, 9, (B, M, K)).astype(np.float64)
    wi = rng.integers(-8, 9, (B, N, K)).astype(np.float64)
    xq, wq = oracle.e4m3_encode(xi), oracle.e4m3_encode(wi)
    xs = np.full((B, M, K // 32), 127, np.uint8)
    ws = np.full((B, N, K // 32), 127, np.uint8)
    pw = ops.process_weights(u8_to_dev(wq if B > 1 else wq[0], dev), u8_to_dev(ws if B > 1 else ws[0], dev))
    xd, sd = u8_to_dev(xq if B > 1 else xq[0], dev), u8_to_dev(xs if B > 1 else xs[0], dev)
    exp = synth.to_bf16_bits(np.matmul(xi, np.swapaxes(wi, 1, 2)))
    for path in (0, 4):
        out = ops.linear(xd, pw, x_scale=sd, path=path)
        ops.check()
        got = bf16_bits(out).reshape(exp.shape)
        assert np.array_equal(got, exp), f"path {path}: {int((got != exp).sum())} mismatches"


@pytest.mark.parametrize("B,M,N,K,bias", [(1, 256, 4096, 4096, True), (1, 200, 1024, 3072, False),
                                          (3, 130, 264, 2048, True), (1, 65, 4096, 4096, True),
                                          (1, 300, 4096, 8192, True)])
def test_against_oracle_and_deterministic(B, M, N, K, bias):
    dev = device()
    assert splits_for(B, M, N, K) > 1
    p = synth.make_problem("splitk", B, M, N, K, seed=M * 3 + K + B, bias_std=0.1 if bias else None)
    wq, ws = oracle_weights(p)
    pw = ops.process_weights(u8_to_dev(wq if B > 1 else wq[0], dev), u8_to_dev(ws if B > 1 else ws[0], dev))
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    b = None if p.bias is None else bf16_to_dev(p.bias, dev)
    a1 = ops.linear(x, pw, b, path=4)
    a2 = ops.linear(x, pw, b, path=4)
    unsplit = ops.linear(x, pw, b, path=3)
    ops.check()
    assert torch.equal(a1.view(torch.int16), a2.view(torch.int16)), "split-K result differs between calls"
    rows = np.arange(M) if M <= 256 else np.arange(0, M, 3)
    xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x[:, rows]))
    ref = oracle.linear(xq, xs, wq, ws, None if p.bias is None else synth.bf16_bits_to_f64(p.bias))
    got = a1 if B > 1 else a1[None]
    assert_close(got[:, rows], ref, f"split-K B={B} M={M} N={N} K={K}")
    from _helpers import tolerance_violations
    u = unsplit.float().cpu().numpy().astype(np.float64).reshape(-1, N)
    s = a1.float().cpu().numpy().astype(np.float64).reshape(-1, N)
    assert not tolerance_violations(s, u).any()


def test_hand_off_through_the_reduce():
    dev = device()
    B, M, N, K = 1, 256, 1024, 4096
    assert splits_for(B, M, N, K) > 1
    p = synth.make_problem("splitk-handoff", B, M, N, K, seed=12, bias_std=0.1)
    wq, ws = oracle_weights(p)
    pw = ops.process_weights(u8_to_dev(wq[0], dev), u8_to_dev(ws[0], dev))
    x, b = bf16_to_dev(p.x[0], dev), bf16_to_dev(p.bias, dev)
    out, y = ops.linear_quantized_out(x, pw, b)
    ref = ops.linear(x, pw, b, path=4)
    ops.check()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    q_ref, s_ref = oracle.quantize(synth.bf16_bits_to_f64(bf16_bits(out))[None])
    assert np.array_equal(y.x_q.cpu().numpy(), q_ref)
    sc = torch.empty((1, M, N // 32), dtype=torch.uint8, device=dev)
    ops._check(ops.load().mxfp8_unpack_scales(y.sf_packed.data_ptr(), 1, M, N, sc.data_ptr(), ops._stream()))
    assert np.array_equal(sc.cpu().numpy(), s_ref)


@pytest.mark.parametrize("fmt", ["e2m3", "e3m2"])
def test_mxfp6_weights_with_split_k(fmt):
    dev = device()
    B, M, N, K = 1, 256, 2048, 4096
    assert splits_for(B, M, N, K) > 1
    p = synth.make_problem("splitk-fp6", B, M, N, K, seed=44, bias_std=0.1)
    wq, ws = ops.quantize_weights(bf16_to_dev(p.w[0], dev), fmt)
    pw = ops.process_weights(wq, ws, fmt)
    x = bf16_to_dev(p.x[0], dev)
    out = ops.linear(x, pw, bf16_to_dev(p.bias, dev))
    ops.check()
    rq, rs = oracle.quantize_fp6(synth.bf16_bits_to_f64(p.w[0]), fmt)
    rows = np.arange(0, M, 4)
    xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x[0, rows]))
    ref = oracle.linear(xq, xs, rq, rs, synth.bf16_bits_to_f64(p.bias), w_format=fmt)
    assert_close(out[rows], ref, f"split-K with {fmt} weights")
