"""mxfp8_linear on the GPU against the oracle.

Exact cases first (integer-valued operands, power-of-two scale patterns: the
fp32 sums are exact, so the bf16 output must equal bf16(oracle) bit for bit),
then tolerance checks on seeded workloads, ragged shapes and the batched form.
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import (assert_close, bf16_bits, bf16_to_dev, device, oracle_weights, u8_to_dev)
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def _pack(wq, ws, dev):
    return ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev))


def _exact_bits(ref):
    """bf16 RNE of an fp64 value that is exact in fp32 (as the GPU rounds it)."""
    return synth.to_bf16_bits(ref)


def _run_prequant(xq, xs, wq, ws, bias=None, path=0):
    dev = device()
    pw = _pack(wq, ws, dev)
    b = None if bias is None else bf16_to_dev(bias, dev)
    out = ops.linear(u8_to_dev(xq, dev), pw, b, x_scale=u8_to_dev(xs, dev), path=path)
    ops.check()
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 256, 512), (256, 512, 4096),
                                   (100, 264, 384), (1, 8, 128)])
def test_integer_operands_exact(M, N, K):
    rng = np.random.default_rng(M + N + K)
    xi = rng.integers(-8, 9, (M, K)).astype(np.float64)
    wi = rng.integers(-8, 9, (N, K)).astype(np.float64)
    xq, wq = oracle.e4m3_encode(xi), oracle.e4m3_encode(wi)
    xs = np.full((M, K // 32), 127, np.uint8)
    ws = np.full((N, K // 32), 127, np.uint8)
    out = _run_prequant(xq, xs, wq, ws)
    ref = xi @ wi.T
    got = bf16_bits(out)
    exp = _exact_bits(ref)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)} mismatches; first {i}: got "
                             f"{synth.bf16_bits_to_f64(np.array([got[i]]))[0]} ref {ref[i]}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (256, 384, 1024), (130, 136, 256)])
def test_power_of_two_scale_patterns_exact(M, N, K):
    """Unit operands with a distinct scale per (row, block): pins the scale layout."""
    KB = K // 32
    m = np.arange(M)[:, None]
    n = np.arange(N)[:, None]
    kb = np.arange(KB)[None, :]
    sx = (127 + (m * 3 + kb * 5) % 7 - 3).astype(np.uint8)
    sw = (127 + (n * 5 + kb * 2) % 9 - 4).astype(np.uint8)
    one = oracle.e4m3_encode(np.ones(1))[0]
    xq = np.full((M, K), one, np.uint8)
    wq = np.full((N, K), one, np.uint8)
    # a sign pattern too, so that a wrong element order cannot cancel out
    xq[:, 1::3] |= 0x80
    out = _run_prequant(xq, sx, wq, sw)
    ref = oracle.linear(xq, sx, wq, sw)
    got = bf16_bits(out)
    exp = _exact_bits(ref)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)}/{got.size} mismatches; first {i}: got "
                             f"{synth.bf16_bits_to_f64(np.array([got[i]]))[0]} ref {ref[i]}")


def test_scale_repack_round_trip():
    dev = device()
    rng = np.random.default_rng(1)
    for B, N, K in [(1, 256, 512), (1, 130, 160), (3, 200, 7168 // 4)]:
        ws = rng.integers(0, 256, (B, N, K // 32)).astype(np.uint8)
        wq = rng.integers(0, 256, (B, N, K)).astype(np.uint8)
        pw = _pack(wq if B > 1 else wq[0], ws if B > 1 else ws[0], dev)
        back = ops.unpack_scales(pw).cpu().numpy()
        assert np.array_equal(back.reshape(B, N, -1), ws)
        assert np.array_equal(pw.w_packed.cpu().numpy(), wq.reshape(-1))
        # the documented atom layout, restated here for the check
        sp = pw.sf_packed.cpu().numpy()
        RT, KT = -(-N // 128), -(-K // 128)
        b, r, k = np.meshgrid(np.arange(B), np.arange(N), np.arange(K // 32), indexing="ij")
        off = ((b * KT + k // 4) * RT + r // 128) * 512 + (r % 128 % 32) * 16 + (r % 128 // 32) * 4 + k % 4
        assert np.array_equal(sp[off], ws)
        mask = np.ones(sp.size, bool)
        mask[off.reshape(-1)] = False
        assert not sp[mask].any(), "padding must be zero"


def _bf16_problem_check(p, path=0, rows=None):
    dev = device()
    wq, ws = oracle_weights(p)
    batched = p.B > 1
    pw = _pack(wq if batched else wq[0], ws if batched else ws[0], dev)
    x = bf16_to_dev(p.x if batched else p.x[0], dev)
    bias = None if p.bias is None else bf16_to_dev(p.bias, dev)
    out = ops.linear(x, pw, bias, path=path)
    ops.check()
    x64 = synth.bf16_bits_to_f64(p.x)
    b64 = None if p.bias is None else synth.bf16_bits_to_f64(p.bias)
    if rows is None:
        xq, xs = oracle.quantize(x64)
        ref = oracle.linear(xq, xs, wq, ws, b64)
        assert_close(out if batched else out[None], ref, p.name)
    else:
        xq, xs = oracle.quantize(x64[0, rows])
        ref = oracle.linear(xq, xs, wq[0], ws[0], b64)
        assert_close(out[rows], ref, p.name + " (sampled rows)")
    return out


def test_tiny():
    _bf16_problem_check(synth.tiny())


@pytest.mark.parametrize("M,N,K,bias", [(1, 8, 128, True), (5, 136, 256, False),
                                        (130, 264, 384, True), (257, 520, 1024, True),
                                        (64, 4096, 512, True)])
def test_ragged_shapes(M, N, K, bias):
    p = synth.make_problem("rag", 1, M, N, K, seed=M * 31 + N, bias_std=0.1 if bias else None)
    _bf16_problem_check(p)


def test_batched_small():
    p = synth.make_problem("bmm-small", 3, 200, 264, 256, seed=8, x_dist="laplace", bias_std=0.1)
    _bf16_problem_check(p)


def test_prequantized_equals_bf16_path():
    dev = device()
    p = synth.make_problem("pq", 1, 300, 512, 1024, seed=13, bias_std=0.1)
    wq, ws = oracle_weights(p)
    pw = _pack(wq[0], ws[0], dev)
    x = bf16_to_dev(p.x[0], dev)
    bias = bf16_to_dev(p.bias, dev)
    a = ops.linear(x, pw, bias)
    xq, xs = ops.quantize(x)
    b = ops.linear(xq, pw, bias, x_scale=xs)
    ops.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("B,M,N,K,path", [(1, 300, 512, 1024, 3), (3, 200, 264, 512, 3), (2, 130, 136, 384, 0),
                                          (1, 256, 1024, 2048, 4), (2, 100, 256, 4096, 4)])
def test_prequantized_scales_read_row_major(B, M, N, K, path):
    """On the CTA-pair kernel (paths 3, 4 and path 0 above 128 rows; path 4
    splits K at these shapes) pre-quantised x goes in with its row-major
    scales, which the kernel's scale writers gather into atom lines
    themselves; bf16 x goes through the quantise kernel's packed atoms.  Same
    kernel, same codes and scales: the outputs must be equal bit for bit
    (ragged rows past M, batches, split-K)."""
    dev = device()
    p = synth.make_problem("rowmajor", B, M, N, K, seed=B + M + N, bias_std=0.1)
    wq, ws = oracle_weights(p)
    pw = _pack(wq if B > 1 else wq[0], ws if B > 1 else ws[0], dev)
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    bias = bf16_to_dev(p.bias, dev)
    xq, xs = ops.quantize(x)
    a = ops.linear(x, pw, bias, path=path)
    b = ops.linear(xq, pw, bias, x_scale=xs, path=path)
    ops.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_leading_dims_flattened():
    dev = device()
    p = synth.make_problem("lead", 1, 2 * 3 * 5, 128, 256, seed=21)
    wq, ws = oracle_weights(p)
    pw = _pack(wq[0], ws[0], dev)
    x = bf16_to_dev(p.x[0], dev)
    out2d = ops.linear(x, pw)
    out3d = ops.linear(x.view(2, 3, 5, 256), pw)
    ops.check()
    assert out3d.shape == (2, 3, 5, 128)
    assert torch.equal(out3d.reshape(30, 128).view(torch.int16), out2d.view(torch.int16))


def test_zero_m_is_noop():
    dev = device()
    p = synth.make_problem("z", 1, 1, 64, 128, seed=1)
    wq, ws = oracle_weights(p)
    pw = _pack(wq[0], ws[0], dev)
    out = ops.linear(torch.empty((0, 128), dtype=torch.bfloat16, device=dev), pw)
    ops.check()
    assert out.shape == (0, 64)


def test_repeated_calls_are_deterministic():
    dev = device()
    p = synth.make_problem("det", 1, 512, 1024, 2048, seed=3, bias_std=0.1)
    wq, ws = oracle_weights(p)
    pw = _pack(wq[0], ws[0], dev)
    x = bf16_to_dev(p.x[0], dev)
    bias = bf16_to_dev(p.bias, dev)
    a = ops.linear(x, pw, bias)
    b = ops.linear(x, pw, bias)
    ops.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ workloads
@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_decode_sweep(M):
    _bf16_problem_check(synth.decode(M))


def _sample_rows(x_bits, M, n_random=96, seed=0):
    x = synth.bf16_bits_to_f64(x_bits[0])
    blocks = x.reshape(M, -1, 32)
    zero_rows = np.nonzero(np.all(blocks == 0, axis=2).any(axis=1))[0][:16]
    outlier_rows = np.nonzero((np.abs(x) > 50).any(axis=1))[0][:16]
    fixed = np.array([0, 1, 127, 128, 129, M // 2, M - 129, M - 128, M - 1])
    rnd = np.random.default_rng(seed).choice(M, n_random, replace=False)
    return np.unique(np.concatenate([fixed, zero_rows, outlier_rows, rnd]))


def test_prefill_up_sampled():
    """The full MLP-up call (the benchmark's configuration and launch) on
    about 512 of its 4096 rows: tile edges, rows with zero blocks and
    outliers, and 480 random rows, every output column."""
    p = synth.prefill_up()
    rows = _sample_rows(p.x, p.M, n_random=480)
    assert len(rows) >= 500
    _bf16_problem_check(p, rows=rows)


def test_prefill_down_prequantized_sampled():
    dev = device()
    p = synth.prefill_down()
    wq, ws = oracle_weights(p)
    x64 = synth.bf16_bits_to_f64(p.x[0])
    del p.x
    xq, xs = oracle.quantize(x64)
    del x64
    pw = _pack(wq[0], ws[0], dev)
    out = ops.linear(u8_to_dev(xq, dev), pw, x_scale=u8_to_dev(xs, dev))
    ops.check()
    rows = np.unique(np.concatenate([[0, 1, 127, 128, p.M - 1],
                                     np.random.default_rng(1).choice(p.M, 507, replace=False)]))
    assert len(rows) >= 500
    ref = oracle.linear(xq[rows], xs[rows], wq[0], ws[0])
    assert_close(out[rows], ref, p.name)


def test_bmm_workload():
    _bf16_problem_check(synth.bmm())


# ------------------------------------------------------------------ small-M path
def _bf16_exact_block_input(M, K, seed):
    """bf16 x whose 32-blocks are +-2^d (d per row and block): quantised exactly."""
    rng = np.random.default_rng(seed)
    d = rng.integers(-3, 4, (M, K // 32))
    sign = rng.choice([-1.0, 1.0], (M, K))
    return sign * np.repeat(np.ldexp(1.0, d), 32, axis=1)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (4, 256, 512), (16, 136, 1024), (33, 264, 256),
                                   (64, 128, 4096), (5, 256, 1536), (40, 136, 3072)])
def test_small_m_path_exact_block_scales(M, N, K):
    """x with a distinct power-of-two block scale per (row, block), integer W:
    exact sums, so the small-M path must equal bf16(oracle) bit for bit.
    K = 1536 and 3072 give each CTA of the K split an odd number (3) of K
    tiles, which the two MMA issuers divide unevenly."""
    dev = device()
    x = _bf16_exact_block_input(M, K, seed=M + K)
    rng = np.random.default_rng(N)
    wi = rng.integers(-8, 9, (N, K)).astype(np.float64)
    wq, ws = oracle.quantize(wi)
    pw = _pack(wq, ws, dev)
    out = ops.linear(bf16_to_dev(synth.to_bf16_bits(x), dev), pw, path=1)
    ops.check()
    xq, xs = oracle.quantize(x)
    ref = oracle.linear(xq, xs, wq, ws)
    got = bf16_bits(out)
    exp = _exact_bits(ref)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        i = tuple(bad[0])
        raise AssertionError(f"{len(bad)}/{got.size} mismatches; first {i}: got "
                             f"{synth.bf16_bits_to_f64(np.array([got[i]]))[0]} ref {ref[i]}")


@pytest.mark.parametrize("M,N,K,bias", [(1, 8, 128, True), (3, 136, 256, False),
                                        (17, 520, 1024, True), (64, 4096, 512, True),
                                        (48, 1000, 7168, True)])
def test_small_m_path_against_oracle(M, N, K, bias):
    p = synth.make_problem("small", 1, M, N, K, seed=M * 7 + N, bias_std=0.1 if bias else None)
    _bf16_problem_check(p, path=1)


def test_small_m_and_large_m_paths_agree():
    dev = device()
    p = synth.make_problem("paths", 1, 40, 1024, 2048, seed=77, bias_std=0.1)
    wq, ws = oracle_weights(p)
    pw = _pack(wq[0], ws[0], dev)
    x = bf16_to_dev(p.x[0], dev)
    bias = bf16_to_dev(p.bias, dev)
    a = ops.linear(x, pw, bias, path=1)
    b = ops.linear(x, pw, bias, path=2)
    ops.check()
    from _helpers import tolerance_violations
    bad = tolerance_violations(a.float().cpu().numpy().astype(np.float64),
                               b.float().cpu().numpy().astype(np.float64))
    assert not bad.any()


def test_small_m_path_refuses_what_it_cannot_do():
    dev = device()
    p = synth.make_problem("refuse", 2, 8, 128, 256, seed=5)
    wq, ws = oracle_weights(p)
    pw = _pack(wq, ws, dev)
    with pytest.raises(ops.MxStatusError) as ei:      # batched
        ops.linear(bf16_to_dev(p.x, dev), pw, path=1)
    assert ei.value.status == 2
    big = synth.make_problem("big", 1, 129, 128, 256, seed=6)
    wq, ws = oracle_weights(big)
    pw = _pack(wq[0], ws[0], dev)
    with pytest.raises(ops.MxStatusError):            # M > 128
        ops.linear(bf16_to_dev(big.x[0], dev), pw, path=1)
    ops.check()


# ------------------------------------------------------------------ CTA-pair tiles at large M
@pytest.mark.parametrize("M,N,K", [(256, 384, 1024), (300, 520, 512), (260, 264, 128), (4096, 4096, 256)])
def test_single_cta_tiles_exact_scales(M, N, K):
    """The large-M path on the exact scale-pattern problem with one CTA per
    128 x 256 tile (path 2) and with 256 x 256 tiles on CTA pairs (path 3).
    K = 128 is one K tile; at 4096 x 4096 x 256 each pair has several tiles of
    two K tiles, so the pair kernel's first ring round spans tile boundaries."""
    KB = K // 32
    m = np.arange(M)[:, None]
    n = np.arange(N)[:, None]
    kb = np.arange(KB)[None, :]
    sx = (127 + (m * 3 + kb * 5) % 7 - 3).astype(np.uint8)
    sw = (127 + (n * 5 + kb * 2) % 9 - 4).astype(np.uint8)
    one = oracle.e4m3_encode(np.ones(1))[0]
    xq = np.full((M, K), one, np.uint8)
    wq = np.full((N, K), one, np.uint8)
    xq[:, 1::3] |= 0x80
    exp = _exact_bits(oracle.linear(xq, sx, wq, sw))
    for path in (2, 3):
        got = bf16_bits(_run_prequant(xq, sx, wq, sw, path=path))
        assert np.array_equal(got, exp), f"path {path}: {int((got != exp).sum())} mismatches"


def test_pair_tiles_ragged_batched_bias():
    p = synth.make_problem("pair-rag", 3, 300, 520, 640, seed=19, bias_std=0.1)
    _bf16_problem_check(p, path=2)
    _bf16_problem_check(p, path=3)
