"""Pins for the oracle's MXFP6 weight path (CPU, no GPU).

The MXFP6 element codecs (E2M3, E3M2) and block quantiser are tied to things
other than themselves: hand-worked blocks (tests/golden/hand_blocks_fp6.txt),
ml_dtypes' float6 types, a nearest-value search over all 64 codes with exact
fractions, the MX property that a block's scaled maximum lands in
[2**emax, 2**(emax+1)), a round-trip bound, brute-force rational GEMMs, and
planted mistakes that some pin must catch.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle.mx_oracle as ox
from mxfp8_block_scaled_02_gb300 import synth
from test_oracle import load_golden

ml_dtypes = pytest.importorskip("ml_dtypes")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks_fp6.txt")
BLOCKS = load_golden(GOLDEN)
FORMATS = ["e2m3", "e3m2"]
ML = {"e2m3": "float6_e2m3fn", "e3m2": "float6_e3m2fn"}


def test_golden_file_is_well_formed():
    assert len(BLOCKS) >= 8
    for b in BLOCKS:
        assert b["format"] in FORMATS and b["x"].shape == (32,) and b["q"].shape == (32,), b["name"]
        assert (b["q"] & 0xC0 == 0).all(), b["name"]                 # 6-bit codes
        fin = np.isfinite(b["x"])
        xb = synth.bf16_bits_to_f64(synth.to_bf16_bits(b["x"][fin]))
        assert np.array_equal(xb, b["x"][fin]), b["name"]


@pytest.mark.parametrize("blk", BLOCKS, ids=[b["name"] for b in BLOCKS])
def test_hand_worked_block(blk):
    q, s = ox.quantize_fp6(blk["x"][None, :], blk["format"])
    assert int(s[0, 0]) == blk["scale"]
    assert np.array_equal(q[0], blk["q"]), [hex(v) for v in q[0]]


# hand-listed positive E2M3 and E3M2 values, codes 0x00..0x1F (from the field
# definitions, written out): E2M3 steps of 1/8 up to 2, 1/4 up to 4, 1/2 up to 7.5
E2M3_POS = [Fraction(i, 8) for i in range(16)] + [Fraction(8 + i, 4) for i in range(8)] + \
           [Fraction(8 + i, 2) for i in range(8)]
# E3M2: subnormals i/16, then binades 1/4, 1/2, 1, 2, 4, 8, 16 with 4 steps each
E3M2_POS = [Fraction(i, 16) for i in range(4)] + \
           [Fraction(4 + i, 4) * Fraction(2) ** (b - 2) for b in range(7) for i in range(4)]


def test_value_tables_by_hand_and_ml_dtypes():
    for fmt, table in (("e2m3", E2M3_POS), ("e3m2", E3M2_POS)):
        assert len(table) == 32
        codes = np.arange(64, dtype=np.uint8)
        v = ox.fp6_value(codes, fmt)
        exp = np.array([float(f) for f in table] + [-float(f) for f in table])
        assert np.array_equal(v, exp) and np.array_equal(np.signbit(v), np.arange(64) >= 32), fmt
        ml = codes.view(getattr(ml_dtypes, ML[fmt])).astype(np.float64)
        assert np.array_equal(ml, v), fmt
        assert ox.fp6_max(fmt) == float(table[-1])


def _dense(fmt):
    """Values on and between every pair of neighbouring codes (ties included),
    well past the largest code, and a random sweep."""
    pos = np.array([float(f) for f in (E2M3_POS if fmt == "e2m3" else E3M2_POS)])
    mids = (pos[1:] + pos[:-1]) / 2
    quarter = np.concatenate([pos[:-1] + (pos[1:] - pos[:-1]) / 4, pos[:-1] + 3 * (pos[1:] - pos[:-1]) / 4])
    big = pos[-1] * np.array([1.0, 1.01, 1.07, 1.5, 2.0, 1e6])
    rnd = np.random.default_rng(3).uniform(0, pos[-1] * 1.2, 20000)
    v = np.concatenate([pos, mids, quarter, big, rnd, np.ldexp(1.0, np.arange(-30, 0))])
    return np.concatenate([v, -v])


def _table_encode(v, fmt):
    """Nearest code by search over all 32 magnitudes; ties to the even code;
    saturating."""
    pos = np.array([float(f) for f in (E2M3_POS if fmt == "e2m3" else E3M2_POS)])
    a = np.minimum(np.abs(v), pos[-1])
    idx = np.searchsorted(pos, a)
    lo, hi = np.clip(idx - 1, 0, 31), np.clip(idx, 0, 31)
    dlo, dhi = a - pos[lo], pos[hi] - a
    pick = np.where(dlo < dhi, lo, hi)
    pick = np.where(dlo == dhi, np.where(lo % 2 == 0, lo, hi), pick)
    return (pick | np.where(np.signbit(v), 0x20, 0)).astype(np.uint8)


@pytest.mark.parametrize("fmt", FORMATS)
def test_encode_matches_table_search_and_ml_dtypes(fmt):
    v = _dense(fmt)
    q = ox.fp6_encode(v, fmt)
    assert np.array_equal(q, _table_encode(v, fmt))
    top = ox.fp6_max(fmt)
    ml = np.clip(v, -top, top).astype(getattr(ml_dtypes, ML[fmt])).view(np.uint8)
    assert np.array_equal(q, ml)
    # every code round-trips
    codes = np.arange(64, dtype=np.uint8)
    assert np.array_equal(ox.fp6_encode(ox.fp6_value(codes, fmt), fmt), codes)


@pytest.mark.parametrize("fmt", FORMATS)
def test_scale_puts_block_max_in_the_top_binade(fmt):
    """For normal blocks, amax / 2**e lies in [2**emax, 2**(emax+1)) exactly."""
    emax = ox.fp6_emax(fmt)
    rng = np.random.default_rng(11)
    x = rng.normal(0, 1, (200, 32)) * np.ldexp(1.0, rng.integers(-60, 60, (200, 1)))
    x = synth.bf16_bits_to_f64(synth.to_bf16_bits(x))
    _, s = ox.quantize_fp6(x, fmt)
    amax = np.abs(x).max(axis=1)
    scaled = np.ldexp(amax, -(s[:, 0].astype(np.int64) - 127))
    assert ((scaled >= 2.0 ** emax) & (scaled < 2.0 ** (emax + 1))).all()


@pytest.mark.parametrize("fmt", FORMATS)
def test_roundtrip_bound(fmt):
    """|x - deq| <= max(2**-(mbits+1) |x|, half a subnormal step * 2**e,
    |x| - max * 2**e) elementwise (nearest rounding with saturation)."""
    _, mbits, bias = ox.FP6_FORMATS[fmt]
    rng = np.random.default_rng(5)
    x = rng.laplace(0, 1, (64, 256)) * np.ldexp(1.0, rng.integers(-20, 20, (64, 1)))
    x = synth.bf16_bits_to_f64(synth.to_bf16_bits(x))
    q, s = ox.quantize_fp6(x, fmt)
    deq = ox.dequantize(q, s, fmt)
    e = np.repeat(s.astype(np.int64) - 127, 32, axis=1)
    err = np.abs(x - deq)
    bound = np.maximum.reduce([np.ldexp(np.abs(x), -(mbits + 1)), np.ldexp(1.0, e + (1 - bias - mbits) - 1),
                               np.abs(x) - ox.fp6_max(fmt) * np.ldexp(1.0, e)])
    assert (err <= bound).all()


def _frac_linear(xq, xs, wq, ws, fmt):
    M, K = xq.shape
    N = wq.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                ex, ew = int(xs[m, k // 32]) - 127, int(ws[n, k // 32]) - 127
                vx = Fraction(float(ox.e4m3_value(xq[m, k]))) * Fraction(2) ** ex
                vw = Fraction(float(ox.fp6_value(wq[n, k], fmt))) * Fraction(2) ** ew
                acc += vx * vw
            out[m, n] = float(acc)
    return out


@pytest.mark.parametrize("fmt", FORMATS)
def test_linear_with_fp6_weights_brute_force(fmt):
    rng = np.random.default_rng(21)
    x = synth.bf16_bits_to_f64(synth.to_bf16_bits(rng.normal(0, 1, (3, 64))))
    w = synth.bf16_bits_to_f64(synth.to_bf16_bits(rng.normal(0, 0.02, (4, 64))))
    xq, xs = ox.quantize(x)
    wq, ws = ox.quantize_fp6(w, fmt)
    ref = ox.linear(xq, xs, wq, ws, w_format=fmt)
    assert np.allclose(ref, _frac_linear(xq, xs, wq, ws, fmt), rtol=0, atol=1e-12 * np.abs(ref).max())
    # and it is not the E4M3 reading of the same bytes
    assert not np.allclose(ref, ox.linear(xq, xs, wq, ws))


# ---------------------------------------------------------------------------
# planted mistakes: each must make some pin above fail
# ---------------------------------------------------------------------------
def _golden_all_pass():
    for b in BLOCKS:
        q, s = ox.quantize_fp6(b["x"][None, :], b["format"])
        if int(s[0, 0]) != b["scale"] or not np.array_equal(q[0], b["q"]):
            return False
    return True


def test_planted_wrong_bias_is_caught(monkeypatch):
    monkeypatch.setitem(ox.FP6_FORMATS, "e2m3", (2, 3, 2))
    assert not _golden_all_pass()


def test_planted_e4m3_emax_is_caught(monkeypatch):
    monkeypatch.setattr(ox, "fp6_emax", lambda fmt: 8)
    assert not _golden_all_pass()


def test_planted_truncation_is_caught(monkeypatch):
    monkeypatch.setattr(ox.np, "rint", np.floor)
    try:
        assert not _golden_all_pass()
    finally:
        monkeypatch.undo()


def test_planted_swapped_formats_are_caught(monkeypatch):
    monkeypatch.setitem(ox.FP6_FORMATS, "e2m3", (3, 2, 3))
    assert not _golden_all_pass()
