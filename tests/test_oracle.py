"""Pins for the CPU oracle: hand-worked blocks, library codecs, brute force.

These run without a GPU.  Each check ties the oracle to something other than
itself: values worked out by hand (tests/golden/hand_blocks.txt), PyTorch's
and ml_dtypes' own FP8 codecs, exact rational arithmetic, integer matmul, and
properties the MX rule fixes (the scaled block maximum lands in [256, 512)).
A last group plants plausible mistakes in a copy of the oracle and checks that
some pin catches each one.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.mx_oracle as ox
from mxfp8_block_scaled_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.txt")


def _expand(tokens, conv):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.rsplit("*", 1)
            out += [conv(v)] * int(n)
        else:
            out.append(conv(t))
    return out


def _float(s):
    s = s.strip()
    if "0x" in s.lower() and "p" in s.lower():
        return float.fromhex(s)
    return float(s)


def load_golden(path=GOLDEN):
    blocks, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("block "):
                cur = {"name": line.split()[1]}
            elif line == "end":
                blocks.append(cur)
                cur = None
            else:
                key, val = line.split(":", 1)
                toks = val.split()
                if key == "x":
                    cur["x"] = np.array(_expand(toks, _float), dtype=np.float64)
                elif key == "scale":
                    cur["scale"] = int(toks[0], 16)
                elif key == "q":
                    cur["q"] = np.array(_expand(toks, lambda t: int(t, 16)), dtype=np.uint8)
                elif key == "format":
                    cur["format"] = toks[0]
    return blocks


GOLDEN_BLOCKS = load_golden()


def test_golden_file_is_well_formed():
    assert len(GOLDEN_BLOCKS) >= 10
    for b in GOLDEN_BLOCKS:
        assert b["x"].shape == (32,), b["name"]
        assert b["q"].shape == (32,), b["name"]
        # every input is exactly representable in bf16
        fin = np.isfinite(b["x"])
        xb = synth.bf16_bits_to_f64(synth.to_bf16_bits(b["x"][fin]))
        assert np.array_equal(xb, b["x"][fin]), b["name"]


@pytest.mark.parametrize("blk", GOLDEN_BLOCKS, ids=[b["name"] for b in GOLDEN_BLOCKS])
def test_hand_worked_block(blk):
    q, s = ox.quantize(blk["x"][None, :])
    assert int(s[0, 0]) == blk["scale"]
    assert np.array_equal(q[0], blk["q"]), [hex(v) for v in q[0]]


# ---------------------------------------------------------------------------
# E4M3 codec against independent implementations
# ---------------------------------------------------------------------------
def _dense_grid():
    """Every fp32 with <= 11 significant bits in [-512, 512] (plus ties of E4M3)."""
    mant = np.arange(1 << 10, 1 << 11, dtype=np.float64)        # 11-bit significands
    vals = [np.ldexp(mant, e) for e in range(-10 - 26, 10 - 10 + 1)]
    v = np.concatenate(vals + [np.array([0.0])])
    v = v[v <= 512.0]
    return np.concatenate([v, -v])


def _table_encode(v):
    """Nearest finite E4M3 by search over all codes; ties to the even code."""
    codes = np.arange(0, 0x7F)
    vals = np.array([_code_value_fraction(int(c)) for c in codes], dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    idx = np.searchsorted(vals, a)                      # vals is increasing
    lo = np.clip(idx - 1, 0, len(vals) - 1)
    hi = np.clip(idx, 0, len(vals) - 1)
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick = np.where(dlo < dhi, lo, hi)
    tie = dlo == dhi
    pick = np.where(tie, np.where(codes[lo] % 2 == 0, lo, hi), pick)
    code = codes[pick].astype(np.int64) | np.where(np.signbit(v), 0x80, 0)
    return code.astype(np.uint8)


def _code_value_fraction(c):
    """E4M3 code value as an exact Fraction, from the field definitions."""
    s = -1 if c & 0x80 else 1
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0:
        return s * Fraction(m, 512)
    return s * Fraction(8 + m, 8) * Fraction(2) ** (e - 7)


def test_e4m3_encode_matches_table_search():
    v = _dense_grid()
    assert np.array_equal(ox.e4m3_encode(v), _table_encode(v))


def test_e4m3_encode_matches_torch_cast():
    v = _dense_grid()
    clamped = np.clip(v, -448.0, 448.0)
    t = torch.from_numpy(clamped.astype(np.float32)).to(torch.float8_e4m3fn)
    ref = t.view(torch.uint8).numpy()
    got = ox.e4m3_encode(v)
    # torch maps -0.0 and +0.0 separately as well; compare all bytes
    assert np.array_equal(got, ref)


def test_e4m3_encode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    v = _dense_grid()
    ref = np.clip(v, -448.0, 448.0).astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ox.e4m3_encode(v), ref)


def test_e4m3_value_matches_torch_and_fractions():
    codes = np.arange(256, dtype=np.uint8)
    got = ox.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    for c in range(256):
        if (c & 0x7F) != 0x7F:
            assert Fraction(got[c]) == _code_value_fraction(c)


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(ox.e4m3_encode(ox.e4m3_value(codes)), codes)


def test_e4m3_special_values():
    v = np.array([np.nan, np.inf, -np.inf, 1e30, -1e30, 448.0, 464.0, 2.0 ** -10,
                  -(2.0 ** -10), 3 * 2.0 ** -10])
    got = ox.e4m3_encode(v)
    assert list(got) == [0x7F, 0x7E, 0xFE, 0x7E, 0xFE, 0x7E, 0x7E, 0x00, 0x80, 0x02]


def test_e8m0_value_matches_torch():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch has no float8_e8m0fnu")
    b = np.arange(256, dtype=np.uint8)
    got = ox.e8m0_value(b)
    ref = torch.from_numpy(b).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[:255], ref[:255])


# ---------------------------------------------------------------------------
# Shared-exponent rule: properties fixed by the definition
# ---------------------------------------------------------------------------
def test_scale_puts_block_max_in_256_512():
    rng = np.random.default_rng(7)
    amax = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-110, 120, 20000))
    e = ox.block_exponent(amax)
    r = amax / np.ldexp(1.0, e)
    assert np.all((r >= 256.0) & (r < 512.0))
    # the same exponent via exact integer arithmetic on the fp64 bits
    bits = amax.view(np.uint64)
    e_bits = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1023 - 8
    assert np.array_equal(e, e_bits)


def test_scale_clamps_and_zero():
    amax = np.array([0.0, 2.0 ** -120, 2.0 ** -119, 2.0 ** -118, 2.0 ** 127, 3.0e38,
                     np.inf, np.nan])
    s = ox.scale_bytes(amax)
    assert list(s) == [0, 0, 0, 1, 246, 246, 255, 255]


def _roundtrip_bound_ok(x, q, s):
    deq = ox.dequantize(q, s)
    e = ox.block_exponent(np.max(np.abs(x.reshape(*x.shape[:-1], -1, 32)), axis=-1))
    pow_e = np.repeat(np.ldexp(1.0, e), 32, axis=-1).reshape(x.shape)
    ax = np.abs(x)
    bound = np.maximum.reduce([2.0 ** -4 * ax, pow_e * 2.0 ** -10, ax - 448.0 * pow_e])
    ok1 = np.abs(x - deq) <= bound
    ok2 = np.abs(deq) <= ax * (1 + 2.0 ** -4) + pow_e * 2.0 ** -10
    same_sign = (np.signbit(deq) == np.signbit(x)) | (deq == 0)
    return ok1 & ok2 & same_sign


@pytest.mark.parametrize("make", [synth.tiny, lambda: synth.make_problem(
    "outliers", 1, 64, 8, 4096, seed=2, outlier_frac=1e-3, zero_block_frac=1e-2),
    lambda: synth.make_problem("lap", 1, 32, 8, 7168, seed=4, x_dist="laplace")])
def test_quantize_roundtrip_bound(make):
    p = make()
    x = synth.bf16_bits_to_f64(p.x)
    q, s = ox.quantize(x)
    assert np.all(_roundtrip_bound_ok(x, q, s))


def test_quantize_bound_scaled_range():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((16, 256)) * np.ldexp(1.0, rng.integers(-130, 120, (16, 1)))
    x = synth.bf16_bits_to_f64(synth.to_bf16_bits(x))
    q, s = ox.quantize(x)
    assert np.all(_roundtrip_bound_ok(x, q, s))


def test_quantize_is_blockwise_and_rowwise_independent():
    p = synth.make_problem("t", 1, 4, 4, 256, seed=5)
    x = synth.bf16_bits_to_f64(p.x[0])
    q, s = ox.quantize(x)
    for r in range(4):
        for kb in range(8):
            qb, sb = ox.quantize(x[r:r + 1, 32 * kb:32 * kb + 32])
            assert sb[0, 0] == s[r, kb]
            assert np.array_equal(qb[0], q[r, 32 * kb:32 * kb + 32])


# ---------------------------------------------------------------------------
# GEMM: brute force, integer exactness, batching
# ---------------------------------------------------------------------------
def _brute_linear(xq, xs, wq, ws, bias):
    M, K = xq.shape
    N = wq.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                sx = Fraction(2) ** (int(xs[m, k // 32]) - 127)
                sw = Fraction(2) ** (int(ws[n, k // 32]) - 127)
                acc += _code_value_fraction(int(xq[m, k])) * sx * _code_value_fraction(int(wq[n, k])) * sw
            if bias is not None:
                acc += Fraction(float(bias[n]))
            out[m][n] = acc
    return out


def test_linear_brute_force_tiny():
    p = synth.make_problem("bf", 1, 3, 5, 96, seed=9, bias_std=0.1)
    x = synth.bf16_bits_to_f64(p.x[0])
    w = synth.bf16_bits_to_f64(p.w[0])
    bias = synth.bf16_bits_to_f64(p.bias)
    xq, xs = ox.quantize(x)
    wq, ws = ox.quantize(w)
    got = ox.linear(xq, xs, wq, ws, bias)
    ref = _brute_linear(xq, xs, wq, ws, bias)
    for m in range(3):
        for n in range(5):
            r = float(ref[m][n])
            assert abs(got[m, n] - r) <= 1e-12 * max(1.0, abs(r))


def test_linear_integer_operands_exact():
    """Integer-valued E4M3 codes with unit scales: the result is an integer matmul."""
    rng = np.random.default_rng(3)
    M, N, K = 7, 9, 256
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    xq = ox.e4m3_encode(xi.astype(np.float64))
    wq = ox.e4m3_encode(wi.astype(np.float64))
    ones_x = np.full((M, K // 32), 127, np.uint8)
    ones_w = np.full((N, K // 32), 127, np.uint8)
    got = ox.linear(xq, ones_x, wq, ones_w)
    assert np.array_equal(got, (xi @ wi.T).astype(np.float64))
    # scales shift each block exactly by its power of two
    sx = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
    sw = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
    exp = np.zeros((M, N))
    for kb in range(K // 32):
        blk = xi[:, 32 * kb:32 * kb + 32] @ wi[:, 32 * kb:32 * kb + 32].T
        exp += blk * np.ldexp(1.0, sx[:, kb:kb + 1].astype(int) - 127) * \
            np.ldexp(1.0, sw[:, kb].astype(int) - 127)[None, :]
    assert np.array_equal(ox.linear(xq, sx, wq, sw), exp)


def test_linear_batched_is_independent_products():
    p = synth.make_problem("b", 3, 4, 8, 128, seed=12, x_dist="laplace", bias_std=0.1)
    x = synth.bf16_bits_to_f64(p.x)
    w = synth.bf16_bits_to_f64(p.w)
    bias = synth.bf16_bits_to_f64(p.bias)
    xq, xs = ox.quantize(x)
    wq, ws = ox.quantize(w)
    out = ox.linear(xq, xs, wq, ws, bias)
    assert out.shape == (3, 4, 8)
    for b in range(3):
        assert np.array_equal(out[b], ox.linear(xq[b], xs[b], wq[b], ws[b], bias))


def test_linear_zero_input_gives_bias():
    K = 64
    xq = np.zeros((2, K), np.uint8)
    xs = np.zeros((2, K // 32), np.uint8)
    wq = ox.e4m3_encode(np.ones((3, K)))
    ws = np.full((3, K // 32), 127, np.uint8)
    bias = np.array([0.5, -2.0, 3.25])
    assert np.array_equal(ox.linear(xq, xs, wq, ws, bias), np.tile(bias, (2, 1)))


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by one of the pins above
# ---------------------------------------------------------------------------
def _golden_all_pass(mod):
    for b in GOLDEN_BLOCKS:
        q, s = mod.quantize(b["x"][None, :])
        if int(s[0, 0]) != b["scale"] or not np.array_equal(q[0], b["q"]):
            return False
    return True


def test_planted_wrong_emax_is_caught(monkeypatch):
    monkeypatch.setattr(ox, "E4M3_EMAX", 7)
    assert not _golden_all_pass(ox)


def test_planted_truncating_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(ox.np, "rint", np.trunc)
    try:
        v = _dense_grid()
        assert not np.array_equal(ox.e4m3_encode(v), _table_encode(v))
    finally:
        monkeypatch.undo()


def test_planted_ties_away_is_caught(monkeypatch):
    monkeypatch.setattr(ox.np, "rint", lambda a: np.floor(np.asarray(a) + 0.5))
    try:
        assert not _golden_all_pass(ox)
    finally:
        monkeypatch.undo()


def test_planted_transposed_weight_is_caught():
    rng = np.random.default_rng(4)
    M = N = 6
    K = 64
    xi = rng.integers(-4, 5, (M, K))
    wi = rng.integers(-4, 5, (N, K))
    one = np.full((M, K // 32), 127, np.uint8)
    xq, wq = ox.e4m3_encode(xi.astype(float)), ox.e4m3_encode(wi.astype(float))
    # the plausible slip: multiplying in the wrong order, W x^T instead of x W^T
    wrong = ox.dequantize(wq, one) @ ox.dequantize(xq, one).T
    assert not np.array_equal(wrong, (xi @ wi.T).astype(float))
    assert np.array_equal(ox.linear(xq, one, wq, one), (xi @ wi.T).astype(float))


def test_planted_missing_sign_is_caught(monkeypatch):
    orig = ox.e4m3_encode
    monkeypatch.setattr(ox, "e4m3_encode", lambda v: orig(np.abs(v)))
    assert not _golden_all_pass(ox)


def test_bf16_max_input_is_finite_in_oracle():
    assert math.isfinite(float.fromhex("0x1.fep127"))
