"""The fused small-M quantiser under an exact check: every rounding case.

The small-M kernel quantises x inside the GEMM, so its codes are seen only
through the product.  With an identity weight (N = K, w[n, k] = 1 if n == k,
one weight scale per K block), out[m, n] = deq(x)[m, n] * 2^s(n): a single
E4M3 value times powers of two, exact in fp32 and in bf16.  So the bf16 output
must equal bf16(oracle) bit for bit, and each output element pins one
quantised element (its code and its block's scale byte).

The eight 32-element K blocks of each row are eight families of cases (the
rows vary exponents and positions inside each family):
  0  round-to-nearest-even ties between E4M3 codes (both directions)
  1  saturation: values in (448, 512) * 2^e, and ties just below 448
  2  E4M3 subnormal results (step 2^-9), with ties on the subnormal grid
  3  all-zero block (+0 and -0 elements): scale byte 0
  4  clamped block: amax below 2^-119 (bf16 normals and subnormals), byte 0
  5  random normal values at several exponents (general rounding)
  6  underflow to signed zero below 2^-10 * 2^e (the tie at 2^-10 -> 0)
  7  large exponents (amax near 2^96)
Weight scales bring every output into the fp32 normal range: +120 for the
clamped block (its scale is 2^-127), -90 for the large-exponent block.
A CPU test checks that the input really contains each case.
"""

import numpy as np
import pytest
import torch

import oracle
from _helpers import bf16_bits, bf16_to_dev, device, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

K = 256
W_SHIFT = [0, 0, 0, 0, 120, 0, 0, -90]   # weight scale exponent per K block


def rounding_input(M: int) -> np.ndarray:
    """[M, 256] fp64 values, every one exactly a bf16 value."""
    x = np.zeros((M, K))
    for m in range(M):
        rng = np.random.default_rng(1000 + m)
        e = (m % 5) - 2
        # 0: ties halfway between consecutive codes, (1 + (2j+1)/16) * 2^E, E in [-6, 7]
        b = x[m, 0:32]
        b[0] = 448.0 * 2.0 ** e
        for i in range(1, 32):
            E = -6 + (i + m) % 14
            j = (i * 3 + m) % 8
            b[i] = (-1) ** i * (1 + (2 * j + 1) / 16) * 2.0 ** (E + e)
        # 1: saturation in (448, 512) * 2^e, ties below 448 (432 -> 448, 400 -> 384)
        b = x[m, 32:64]
        sat = [450, 456, 464, 480, 496, 504, 510, 449.0 + 7]
        below = [432, 400, 368, 336, 440, 447, 446]
        vals = sat + below
        for i in range(32):
            v = vals[(i + m) % len(vals)]
            b[i] = (-1) ** (i // 3) * v * 2.0 ** e
        # 2: subnormal results: amax 256 * 2^e, others k * 2^-10 * 2^e, k in 1..31
        b = x[m, 64:96]
        b[0] = 256.0 * 2.0 ** e
        for i in range(1, 32):
            k = (i + 5 * m) % 31 + 1
            b[i] = (-1) ** (i + m) * k * 2.0 ** (-10 + e)
        # 3: zero block with signed zeros
        x[m, 96:128] = np.where(np.arange(32) % 3 == 0, -0.0, 0.0)
        # 4: clamped: amax < 2^-119; bf16 normals near 2^-124 and subnormals 2^-127..2^-133
        b = x[m, 128:160]
        for i in range(32):
            if i % 2 == 0:
                b[i] = (1 + ((i + m) % 8) / 8) * 2.0 ** (-124 - (i + m) % 3)
            else:
                b[i] = ((i + m) % 7 + 1) * 2.0 ** (-133 + (i % 4))
            if i % 5 == 0:
                b[i] = -b[i]
        # 5: random normal values
        x[m, 160:192] = rng.normal(0.0, 1.0, 32) * 2.0 ** ((m % 7) - 3)
        # 6: underflow to signed zero: amax 300 * 2^e; tiny values at and below 2^-10 * 2^e
        b = x[m, 192:224]
        b[0] = 300.0 * 2.0 ** e
        for i in range(1, 32):
            b[i] = (-1) ** i * 2.0 ** (-10 - (i + m) % 6 + e)
        # 7: large exponents
        x[m, 224:256] = rng.normal(0.0, 1.0, 32) * 2.0 ** 95
    x = synth.bf16_bits_to_f64(synth.to_bf16_bits(x))   # bf16 values (exact for the constructed ones)
    return x


def identity_weights():
    one = oracle.e4m3_encode(np.ones(1))[0]
    wq = np.zeros((K, K), np.uint8)
    wq[np.arange(K), np.arange(K)] = one
    ws = np.empty((K, K // 32), np.uint8)
    for n in range(K):
        ws[n, :] = 127 + W_SHIFT[n // 32]
    return wq, ws


def test_rounding_input_covers_every_case():
    """CPU: the constructed input contains each rounding case (per the oracle)."""
    x = rounding_input(64)
    exact = synth.bf16_bits_to_f64(synth.to_bf16_bits(x))
    assert np.array_equal(exact, x)
    xq, xs = oracle.quantize(x)
    blk = xq.reshape(64, 8, 32)
    e = xs.astype(np.int64) - 127
    scaled = np.ldexp(x.reshape(64, 8, 32), -e[..., None])
    code_val = oracle.e4m3_value(blk)
    # 0: ties (exactly halfway) that RNE resolved to an even mantissa
    d = np.abs(scaled[:, 0]) - np.abs(code_val[:, 0])
    assert (np.abs(d[:, 1:]) > 0).all() and ((blk[:, 0, 1:] & 1) == 0).all()
    # 1: saturated values above 448 and ties at 432 -> 448
    assert ((np.abs(scaled[:, 1]) > 448) & ((blk[:, 1] & 0x7F) == 0x7E)).sum() > 64
    assert ((np.abs(scaled[:, 1]) == 432) & ((blk[:, 1] & 0x7F) == 0x7E)).any()
    # 2: subnormal codes (exponent field 0, mantissa != 0)
    assert (((blk[:, 2] >> 3) & 0xF) == 0).sum() > 64 and ((blk[:, 2] & 7) != 0).sum() > 64
    # 3, 4: scale byte 0 (zero block and clamped block)
    assert (xs[:, 3] == 0).all() and (xs[:, 4] == 0).all()
    assert (blk[:, 4] != 0).any()                      # clamped blocks still carry codes
    # 6: values at or below 2^-10 * 2^e become signed zeros
    assert ((blk[:, 6, 1:] & 0x7F) == 0).all() and (blk[:, 6, 1:] == 0x80).any()
    # 7: large exponents
    assert (xs[:, 7] > 127 + 80).all()
    # every output of the identity product is exact in bf16
    wq, ws = identity_weights()
    ref = oracle.linear(xq, xs, wq, ws)
    nz = ref != 0
    assert np.array_equal(synth.bf16_bits_to_f64(synth.to_bf16_bits(ref)), ref)
    assert (np.abs(ref[nz]) >= 2.0 ** -126).all()     # fp32 normal range


def _zero_sign_free(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns with -0 mapped to +0 (the sign of a zero sum is not
    part of the contract: it depends on the order of the zero products)."""
    b = bits.copy()
    b[b == 0x8000] = 0
    return b


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 5, 16, 33, 64])
def test_fused_quantiser_rounding_is_exact(M):
    dev = device()
    x = rounding_input(M)
    wq, ws = identity_weights()
    pw = ops.process_weights(u8_to_dev(wq, dev), u8_to_dev(ws, dev))
    xd = bf16_to_dev(synth.to_bf16_bits(x), dev)
    xq, xs = oracle.quantize(x)
    exp = _zero_sign_free(synth.to_bf16_bits(oracle.linear(xq, xs, wq, ws)))
    outs = {}
    for path in (1, 2, 3, 5):                    # fused small-M, one-CTA, CTA-pair, fused large-M
        out = ops.linear(xd, pw, path=path)
        ops.check()
        got = _zero_sign_free(bf16_bits(out))
        if not np.array_equal(got, exp):
            bad = np.argwhere(got != exp)
            i = tuple(bad[0])
            raise AssertionError(
                f"path {path}: {len(bad)}/{got.size} mismatches; first {i} (K block {i[1] // 32}): got "
                f"{synth.bf16_bits_to_f64(np.array([got[i]]))[0]!r} ref "
                f"{synth.bf16_bits_to_f64(np.array([exp[i]]))[0]!r}")
        outs[path] = got
    # the fused quantisers and the standalone one give bit-identical outputs
    assert np.array_equal(outs[1], outs[2]) and np.array_equal(outs[2], outs[3])
    assert np.array_equal(outs[5], outs[2])
    # and the standalone quantiser's codes and scales are the oracle's
    q, s = ops.quantize(xd)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), xq) and np.array_equal(s.cpu().numpy(), xs)
