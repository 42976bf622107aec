"""The seeded input generator: published SplitMix64 outputs, determinism, shape and value recipes."""

import numpy as np

from mxfp8_block_scaled_02_gb300 import synth


def test_splitmix64_published_outputs():
    # First three outputs of SplitMix64 started from state 0 (the reference
    # values published with the generator by Vigna, prng.di.unimi.it).
    got = [int(v) for v in synth.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_deterministic_and_offsettable():
    a = synth.splitmix64(7, 0, 100)
    b = synth.splitmix64(7, 40, 60)
    assert np.array_equal(a[40:], b)
    assert np.array_equal(synth.normal(3, 1001), synth.normal(3, 1001))


def test_distributions():
    z = synth.normal(1, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    lap = synth.laplace(4, 400000)
    assert abs(lap.mean()) < 0.01 and abs(np.abs(lap).mean() - 1) < 0.01
    u = synth.uniform(5, 0, 100000)
    assert u.min() > 0 and u.max() < 1


def test_bf16_rounding_is_rne():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40])
    bits = synth.to_bf16_bits(v)
    back = synth.bf16_bits_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert list(back[:4]) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5]
    assert back[4] > 0


def test_prefill_up_recipe_small():
    p = synth.make_problem("t", 1, 64, 8, 4096, seed=2, outlier_frac=1e-3, zero_block_frac=1e-2)
    x = synth.bf16_bits_to_f64(p.x).reshape(-1, 32)
    zero_blocks = np.all(x == 0, axis=1).mean()
    assert 0.004 < zero_blocks < 0.02
    assert np.abs(x).max() > 50          # outliers x100 of N(0,1)
    assert p.x.dtype == np.uint16 and p.x.shape == (1, 64, 4096)


def test_workload_shapes():
    t = synth.tiny()
    assert (t.B, t.M, t.N, t.K) == (1, 16, 256, 512) and t.bias is None
    d = synth.make_problem("d", 1, 4, 64, 128, seed=1, bias_std=0.1)
    assert d.bias.shape == (64,)
