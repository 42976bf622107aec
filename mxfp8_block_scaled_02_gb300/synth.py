"""Seeded synthetic inputs for the MXFP8 linear layer.

This module draws the bf16 activations, weights and biases that the tests and
the benchmark feed to both the CUDA path and the CPU oracle.  It holds none of
the quantisation or GEMM arithmetic: it only produces bf16 bit patterns.

Generator (fixed, so data are bit-reproducible on any host and any numpy):

* ``splitmix64``: the i-th draw of stream ``seed`` is the SplitMix64 output
  for state ``seed + (i + 1) * 0x9E3779B97F4A7C15`` (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* uniform on (0, 1): ``((u64 >> 11) + 0.5) * 2**-53``.
* normal: Box-Muller on consecutive pairs of uniforms (u1, u2):
  ``r = sqrt(-2 ln u1)``, ``(r cos 2 pi u2, r sin 2 pi u2)``.
* Laplace(0, b): inverse CDF, ``-b * sign(u - 1/2) * ln(1 - 2 |u - 1/2|)``.
* bf16: fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest even
  on the fp32 bit pattern).

Stream assignment per workload: x uses ``seed``, the bf16 weights ``seed +
1000`` and the bias ``seed + 2000``; structural draws (outlier positions and
zeroed blocks) use ``seed + 3000`` and ``seed + 4000``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of SplitMix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform(seed: int, start: int, count: int) -> np.ndarray:
    """Uniform fp64 on the open interval (0, 1)."""
    u = splitmix64(seed, start, count) >> np.uint64(11)
    return (u.astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, count: int, std: float = 1.0) -> np.ndarray:
    """``count`` N(0, std^2) draws in fp64 (Box-Muller, both outputs kept)."""
    out = np.empty(count, dtype=np.float64)
    pairs = (count + 1) // 2
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        u = uniform(seed, 2 * p0, 2 * (p1 - p0))
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        n = min(count - 2 * p0, z.size)
        out[2 * p0:2 * p0 + n] = z[:n]
    return out * std


def laplace(seed: int, count: int, b: float = 1.0) -> np.ndarray:
    """``count`` Laplace(0, b) draws in fp64 (inverse CDF)."""
    out = np.empty(count, dtype=np.float64)
    for s0 in range(0, count, _CHUNK):
        s1 = min(count, s0 + _CHUNK)
        d = uniform(seed, s0, s1 - s0) - 0.5
        out[s0:s1] = -np.sign(d) * np.log1p(-2.0 * np.abs(d))
    return out * b


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE) bit patterns as uint16.

    Non-finite values are not produced by this module and are not handled.
    """
    f = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    lsb = (f >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = f + np.uint32(0x7FFF) + lsb
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (NaN patterns stay NaN)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns raise the flag on widening
        return b.view(np.float32).astype(np.float64)


@dataclasses.dataclass
class LinearProblem:
    """One synthetic problem: bf16 bit patterns for x, the weights and bias.

    ``x`` is ``[B, M, K]``, ``w`` is ``[B, N, K]`` (both uint16 bf16 bits,
    row-major), ``bias`` is ``[N]`` or None.  ``prequantized`` says that the
    workload hands the layer an already-quantised activation (the caller
    quantises ``x`` once, outside the timed region).
    """

    name: str
    B: int
    M: int
    N: int
    K: int
    x: np.ndarray
    w: np.ndarray
    bias: np.ndarray | None
    prequantized: bool = False

    @property
    def flops(self) -> float:
        return 2.0 * self.B * self.M * self.N * self.K


def _outliers_and_zero_blocks(x: np.ndarray, seed: int, outlier_frac: float,
                              outlier_mult: float, zero_block_frac: float) -> None:
    """In place on fp64 ``x``: scale a fraction of entries, zero 32-blocks.

    Positions are drawn uniformly (with replacement) from their own streams,
    ``seed + 3000`` for outliers and ``seed + 4000`` for zeroed blocks.
    """
    flat = x.reshape(-1)
    n_out = int(round(flat.size * outlier_frac))
    if n_out:
        idx = (uniform(seed + 3000, 0, n_out) * flat.size).astype(np.int64)
        flat[idx] *= outlier_mult
    blocks = flat.reshape(-1, 32)
    n_zero = int(round(blocks.shape[0] * zero_block_frac))
    if n_zero:
        idx = (uniform(seed + 4000, 0, n_zero) * blocks.shape[0]).astype(np.int64)
        blocks[idx, :] = 0.0


def make_problem(name: str, B: int, M: int, N: int, K: int, seed: int, *,
                 x_dist: str = "normal", x_std: float = 1.0, w_std: float = 0.02,
                 bias_std: float | None = None, outlier_frac: float = 0.0,
                 outlier_mult: float = 100.0, zero_block_frac: float = 0.0,
                 prequantized: bool = False) -> LinearProblem:
    if x_dist == "normal":
        xv = normal(seed, B * M * K, x_std)
    elif x_dist == "laplace":
        xv = laplace(seed, B * M * K, x_std)
    else:
        raise ValueError(x_dist)
    if outlier_frac or zero_block_frac:
        _outliers_and_zero_blocks(xv, seed, outlier_frac, outlier_mult, zero_block_frac)
    x = to_bf16_bits(xv).reshape(B, M, K)
    del xv
    w = to_bf16_bits(normal(seed + 1000, B * N * K, w_std)).reshape(B, N, K)
    bias = None
    if bias_std is not None:
        bias = to_bf16_bits(normal(seed + 2000, N, bias_std))
    return LinearProblem(name, B, M, N, K, x, w, bias, prequantized)


# The five workloads of the layer, with their shapes and value recipes.
def tiny() -> LinearProblem:
    return make_problem("tiny M16 N256 K512", 1, 16, 256, 512, seed=0)


def decode(M: int) -> LinearProblem:
    return make_problem(f"decode M{M} N4096 K4096", 1, M, 4096, 4096, seed=1,
                        bias_std=0.1)


def prefill_up() -> LinearProblem:
    return make_problem("prefill MLP-up M4096 N14336 K4096", 1, 4096, 14336, 4096,
                        seed=2, outlier_frac=1e-3, outlier_mult=100.0,
                        zero_block_frac=1e-2)


def prefill_down() -> LinearProblem:
    return make_problem("prefill MLP-down pre-quantized M8192 N4096 K14336", 1, 8192,
                        4096, 14336, seed=3, w_std=0.01, prequantized=True)


def bmm() -> LinearProblem:
    return make_problem("bmm B16 M512 N512 K7168", 16, 512, 512, 7168, seed=4,
                        x_dist="laplace")


WORKLOADS = {
    "tiny": tiny,
    "decode1": lambda: decode(1),
    "decode4": lambda: decode(4),
    "decode16": lambda: decode(16),
    "decode64": lambda: decode(64),
    "prefill_up": prefill_up,
    "prefill_down": prefill_down,
    "bmm": bmm,
}
