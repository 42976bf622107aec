"""MXFP6 weights on the GPU (the mxfp6 page's E2M3 / E3M2 weights with MXFP8
activations, multiplied by the same kind::mxf8f6f4 tensor-core MMA).

* the weight quantiser equals oracle.quantize_fp6 bit for bit (hand-worked
  blocks, every bf16 pattern, every value on the format's grid);
* the packed 6-bit layout is the documented one (restated here);
* the GEMM is exact where the fp32 sums are exact (integer operands, unit
  operands with power-of-two scale patterns) on all three kernel paths, and
  within the parity tolerance of oracle.linear(..., w_format) on seeded
  problems, ragged and batched shapes;
* weights restored from a blob give the same output bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_close, bf16_bits, bf16_to_dev, device, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth
from test_oracle import load_golden
from test_oracle_fp6 import GOLDEN as GOLDEN_FP6

pytestmark = pytest.mark.gpu
FORMATS = ["e2m3", "e3m2"]


def _gpu_quantize(bits: np.ndarray, fmt: str):
    dev = device()
    q, s = ops.quantize_weights(bf16_to_dev(bits, dev), fmt)
    ops.check()
    return q.cpu().numpy(), s.cpu().numpy()


def _assert_exact(bits: np.ndarray, fmt: str):
    q, s = _gpu_quantize(bits, fmt)
    rq, rs = oracle.quantize_fp6(synth.bf16_bits_to_f64(bits), fmt)
    assert np.array_equal(s, rs), f"{int((s != rs).sum())} scale bytes differ"
    if not np.array_equal(q, rq):
        bad = np.argwhere(q != rq)[:5]
        raise AssertionError(f"{fmt}: {int((q != rq).sum())} codes differ, first at {bad.tolist()}: "
                             f"gpu {[hex(q[tuple(i)]) for i in bad]} oracle {[hex(rq[tuple(i)]) for i in bad]}")


def test_hand_worked_fp6_blocks_on_gpu():
    for b in load_golden(GOLDEN_FP6):
        q, s = _gpu_quantize(synth.to_bf16_bits(b["x"][None, :]), b["format"])
        assert int(s[0, 0]) == b["scale"], (b["name"], hex(s[0, 0]))
        assert np.array_equal(q[0], b["q"]), (b["name"], [hex(v) for v in q[0]])


@pytest.mark.parametrize("fmt", FORMATS)
def test_every_bf16_pattern(fmt):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    _assert_exact(allbits.reshape(-1, 1024), fmt)
    perm = (np.arange(65536, dtype=np.int64) * 40503) % 65536
    _assert_exact(allbits[perm].reshape(-1, 2048), fmt)


@pytest.mark.parametrize("fmt", FORMATS)
def test_rounding_grid_at_unit_scale(fmt):
    """Blocks led by 2**emax (scale 2^0), filled with every bf16 value up to 2**(emax+1)."""
    emax = oracle.fp6_emax(fmt)
    top = synth.to_bf16_bits(np.array([2.0 ** (emax + 1)]))[0]
    b = np.arange(0, int(top), dtype=np.uint16)
    v = np.concatenate([b, b | np.uint16(0x8000)])
    pad = (-v.size) % 31
    v = np.concatenate([v, np.zeros(pad, np.uint16)]).reshape(-1, 31)
    lead = np.full((v.shape[0], 1), synth.to_bf16_bits(np.array([2.0 ** emax]))[0], np.uint16)
    _assert_exact(np.concatenate([lead, v], axis=1), fmt)


def _pack6(codes: np.ndarray) -> np.ndarray:
    """The packed 6-bit layout, restated: every 16 codes -> 12 bytes, code i in
    bits [6i, 6i + 6) of the little-endian 96-bit group."""
    c = codes.reshape(-1, 16).astype(np.uint64) & 0x3F
    lo = np.zeros(c.shape[0], np.uint64)
    hi = np.zeros(c.shape[0], np.uint64)
    for i in range(16):
        bit = 6 * i
        if bit + 6 <= 64:
            lo |= c[:, i] << np.uint64(bit)
        elif bit >= 64:
            hi |= c[:, i] << np.uint64(bit - 64)
        else:                                           # straddles the 64-bit boundary
            lo |= (c[:, i] << np.uint64(bit)) & np.uint64(0xFFFFFFFFFFFFFFFF)
            hi |= c[:, i] >> np.uint64(64 - bit)
    out = np.zeros((c.shape[0], 12), np.uint8)
    for j in range(8):
        out[:, j] = ((lo >> np.uint64(8 * j)) & np.uint64(0xFF)).astype(np.uint8)
    for j in range(4):
        out[:, 8 + j] = ((hi >> np.uint64(8 * j)) & np.uint64(0xFF)).astype(np.uint8)
    return out.reshape(-1)


@pytest.mark.parametrize("fmt", FORMATS)
def test_packed_layout(fmt):
    dev = device()
    rng = np.random.default_rng(7)
    B, N, K = 2, 40, 256
    codes = rng.integers(0, 64, (B, N, K)).astype(np.uint8)
    scales = rng.integers(100, 150, (B, N, K // 32)).astype(np.uint8)
    pw = ops.process_weights(u8_to_dev(codes, dev), u8_to_dev(scales, dev), fmt)
    torch.cuda.synchronize()
    assert pw.w_packed.numel() == B * N * K * 3 // 4
    assert np.array_equal(pw.w_packed.cpu().numpy(), _pack6(codes))
    assert np.array_equal(ops.unpack_scales(pw).cpu().numpy(), scales)


def _exact_bits(ref):
    return synth.to_bf16_bits(ref)


def _run(xq, xs, wq, ws, fmt, path, bias=None):
    dev = device()
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev), fmt)
    b = None if bias is None else bf16_to_dev(bias, dev)
    out = ops.linear(u8_to_dev(xq, dev), pw, b, x_scale=u8_to_dev(xs, dev), path=path)
    ops.check()
    return out


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (300, 384, 1024), (1, 128, 512), (64, 136 * 2, 384)])
def test_integer_operands_exact(fmt, M, N, K):
    """Integer activations |x| <= 8 (E4M3) and integer weights |w| <= 7 (exact
    in both FP6 formats), all scales 2^0: every fp32 sum is exact."""
    rng = np.random.default_rng(M + N + K)
    xi = rng.integers(-8, 9, (M, K)).astype(np.float64)
    wi = rng.integers(-7, 8, (N, K)).astype(np.float64)
    xq, wq = oracle.e4m3_encode(xi), oracle.fp6_encode(wi, fmt)
    assert np.array_equal(oracle.fp6_value(wq, fmt), wi)
    xs = np.full((M, K // 32), 127, np.uint8)
    ws = np.full((N, K // 32), 127, np.uint8)
    exp = _exact_bits(xi @ wi.T)
    for path in (2, 3):
        got = bf16_bits(_run(xq, xs, wq, ws, fmt, path))
        assert np.array_equal(got, exp), f"{fmt} path {path}: {int((got != exp).sum())} mismatches"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (16, 128, 1024), (40, 256, 384), (100, 256, 1024),
                                   (128, 128, 512)])
def test_small_m_path_exact(fmt, M, N, K):
    """The fused small-M kernel (weights on the MMA's A side): x = +-2^d per
    block (quantised without rounding), integer FP6 weights: exact sums."""
    dev = device()
    rng = np.random.default_rng(M * 3 + K)
    d = rng.integers(-3, 4, (M, K // 32))          # sums stay within 24 bits
    x = rng.choice([-1.0, 1.0], (M, K)) * np.repeat(np.ldexp(1.0, d), 32, axis=1)
    wi = rng.integers(-7, 8, (N, K)).astype(np.float64)
    wq, ws = oracle.quantize_fp6(wi, fmt)
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev), fmt)
    out = ops.linear(bf16_to_dev(synth.to_bf16_bits(x), dev), pw, path=1)
    ops.check()
    xq, xs = oracle.quantize(x)
    ref = oracle.linear(xq, xs, wq, ws, w_format=fmt)
    got = bf16_bits(out)
    exp = _exact_bits(ref)
    assert np.array_equal(got, exp), f"{fmt}: {int((got != exp).sum())} mismatches"


@pytest.mark.parametrize("fmt", FORMATS)
def test_power_of_two_scale_patterns_exact(fmt):
    """Unit operands with a distinct scale per (row, block): pins the scale
    layout with FP6 weights on every path."""
    M, N, K = 130, 264, 512
    KB = K // 32
    m, n, kb = np.arange(M)[:, None], np.arange(N)[:, None], np.arange(KB)[None, :]
    sx = (127 + (m * 3 + kb * 5) % 7 - 3).astype(np.uint8)
    sw = (127 + (n * 5 + kb * 2) % 9 - 4).astype(np.uint8)
    xq = np.full((M, K), oracle.e4m3_encode(np.ones(1))[0], np.uint8)
    xq[:, 1::3] |= 0x80
    wq = np.full((N, K), oracle.fp6_encode(np.ones(1), fmt)[0], np.uint8)
    exp = _exact_bits(oracle.linear(xq, sx, wq, sw, w_format=fmt))
    for path in (2, 3):
        got = bf16_bits(_run(xq, sx, wq, sw, fmt, path))
        assert np.array_equal(got, exp), f"{fmt} path {path}: {int((got != exp).sum())} mismatches"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("B,M,N,K,path", [(1, 1, 4096, 4096, 0), (1, 16, 4096, 1024, 0), (1, 64, 520, 512, 0),
                                          (1, 300, 520, 1024, 0), (1, 129, 264, 384, 2), (3, 200, 264, 256, 0),
                                          (1, 4096, 1024, 512, 3), (1, 128, 520, 1024, 0)])
def test_against_oracle(fmt, B, M, N, K, path):
    """Seeded bf16 x quantised in the call, weights from bf16 N(0, 0.02)
    quantised to FP6 by the library, bias; every kernel path and a batch."""
    dev = device()
    p = synth.make_problem(f"fp6-{fmt}", B, M, N, K, seed=M + N + K + B, bias_std=0.1)
    w = bf16_to_dev(p.w if B > 1 else p.w[0], dev)
    wq, ws = ops.quantize_weights(w, fmt)
    pw = ops.process_weights(wq, ws, fmt)
    x = bf16_to_dev(p.x if B > 1 else p.x[0], dev)
    out = ops.linear(x, pw, bf16_to_dev(p.bias, dev), path=path)
    ops.check()
    rq, rs = oracle.quantize_fp6(synth.bf16_bits_to_f64(p.w), fmt)
    assert np.array_equal(wq.cpu().numpy().reshape(rq.shape), rq)
    rows = np.arange(M) if M <= 512 else np.arange(0, M, 16)
    xq, xs = oracle.quantize(synth.bf16_bits_to_f64(p.x[:, rows]))
    ref = oracle.linear(xq, xs, rq, rs, synth.bf16_bits_to_f64(p.bias), w_format=fmt)
    got = out if B > 1 else out[None]
    assert_close(got[:, rows], ref, f"{fmt} B={B} M={M} N={N} K={K} path={path}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_blob_round_trip_fp6(fmt):
    dev = device()
    p = synth.make_problem("fp6-blob", 1, 64, 512, 512, seed=9, bias_std=0.1)
    wq, ws = ops.quantize_weights(bf16_to_dev(p.w[0], dev), fmt)
    pw = ops.process_weights(wq, ws, fmt)
    back = ops.load_packed(ops.save_packed(pw), dev)
    assert back.fmt == fmt
    x = bf16_to_dev(p.x[0], dev)
    a, b = ops.linear(x, pw), ops.linear(x, back)
    ops.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
