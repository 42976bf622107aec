"""CPU oracle for the W8A8 MXFP8 linear layer.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The library never calls it and shares
no code with it: nothing here is used by the CUDA path, and nothing here
imports the CUDA path.

Plain, slow and meant to be checked by eye.  All floating point is fp64.

What the layer computes (sources):

* "CompressedTensorsW8A8Mxfp8" (compressed_tensors_w8a8_mxfp8 page), class
  docstring "MXFP8 format": elements are FP8 E4M3 (``float8_e4m3fn``), each
  group of 32 consecutive elements along K shares one uint8 E8M0 scale, and
  activations are quantised dynamically at run time.
* same page, ``create_weights``: weight ``[N, K]`` E4M3 and weight_scale
  ``[N, K // 32]`` uint8.
* "AiterFlyDSLMxfp8LinearKernel" (aiter_flydsl page), class docstring and
  ``apply_weights``: activation scales are row-major ``[M, K // 32]``; the
  output is ``x_q`` times the weight (both dequantised by their block scales),
  in the input dtype, reshaped to ``[*lead, N]``, then ``+ bias``.
* "Mxfp8LinearLayerConfig" (Mxfp8LinearKernel page): ``bmm_batch_size``
  selects a batched layer; read here as B independent products.
* "MxFp6LinearLayerConfig" (mxfp6 page): weights quantised per block of 32
  with weight_quant_key kMxfp6E2M3Static or kMxfp6E3M2Static, i.e. FP6 E2M3 or
  E3M2 elements with the same E8M0 block scales; used here with MXFP8
  activations (``linear(..., w_format=...)``).

The pages name ``mxfp8_e4m3_quantize`` but never show its arithmetic.  The
rule used below is the OCP Microscaling Formats (MX) v1.0 conversion
(section 6.3): shared exponent = floor(log2(amax of the block)) - emax(E4M3),
emax(E4M3) = 8 because the largest finite E4M3 value is 448 = 1.75 * 2**8;
the exponent is clamped to the E8M0 range and each element x / 2**e is rounded
to E4M3 with round-to-nearest-even and saturation to +-448.

Conventions where the pages and the spec leave a choice (each one is pinned by
a test):

* all-zero block: scale byte 0 (exponent -127), elements keep their sign.
* block with a NaN or Inf: scale byte 0xFF (E8M0 NaN), every element 0x7F.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32            # MXFP8 block size along K ("group_size=32")
E4M3_EMAX = 8         # floor(log2(448))
E4M3_MAX = 448.0
E8M0_BIAS = 127
E8M0_NAN = 0xFF
E4M3_NAN = 0x7F


# --------------------------------------------------------------------------
# E8M0 shared exponent (OCP MX v1.0, section 6.3)
# --------------------------------------------------------------------------
def block_exponent(amax: np.ndarray, emax: int | None = None) -> np.ndarray:
    """Unbiased shared exponent e per block, from the block amax (fp64).

    e = floor(log2(amax)) - emax (8 for E4M3), taken exactly from frexp
    (amax = f * 2**ex with f in [0.5, 1), so floor(log2(amax)) = ex - 1),
    clamped to [-127, 127].  A zero block has log2(0) = -inf and clamps to
    -127.  Non-finite amax is returned as 0 here; :func:`scale_bytes` marks
    those blocks as NaN.
    """
    if emax is None:
        emax = E4M3_EMAX
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(np.where(np.isfinite(amax), amax, 0.0))
    e = (ex.astype(np.int64) - 1) - emax
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127)


def scale_bytes(amax: np.ndarray, emax: int | None = None) -> np.ndarray:
    """E8M0 scale byte per block: e + 127, or 0xFF for a non-finite block."""
    b = block_exponent(amax, emax) + E8M0_BIAS
    b = np.where(np.isfinite(amax), b, E8M0_NAN)
    return b.astype(np.uint8)


def e8m0_value(byte: np.ndarray) -> np.ndarray:
    """2**(byte - 127); byte 0xFF is NaN."""
    byte = np.asarray(byte).astype(np.int64)
    v = np.ldexp(1.0, byte - E8M0_BIAS)
    return np.where(byte == E8M0_NAN, np.nan, v)


# --------------------------------------------------------------------------
# FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN, max finite 448)
# --------------------------------------------------------------------------
def e4m3_value(code: np.ndarray) -> np.ndarray:
    """Value of an E4M3 code: exponent bias 7, subnormals m * 2**-9."""
    c = np.asarray(code).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp((8 + m).astype(np.float64), ef - 10)   # (1 + m/8) * 2**(ef-7)
    sub = np.ldexp(m.astype(np.float64), -9)
    v = np.where(ef == 0, sub, normal)
    v = np.where((ef == 15) & (m == 7), np.nan, v)
    return s * v


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to E4M3 codes: nearest, ties to even, saturating.

    |v| >= 448 (Inf included) gives +-448 (0x7E / 0xFE); NaN gives 0x7F.
    Below 2**-6 the grid is the subnormal one, step 2**-9; from 2**E
    (E >= -6) up to 2**(E+1) the step is 2**(E-3).  The sign is kept, so a
    value that rounds to zero gives 0x00 or 0x80.
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(v)
    a_fin = np.where(nan | (a >= E4M3_MAX), 0.0, a)

    # subnormal range: q = a / 2**-9 rounded; q == 8 is the code of 2**-6
    q_sub = np.rint(np.ldexp(a_fin, 9)).astype(np.int64)

    # normal range: a = f * 2**ex, f in [0.5, 1)  =>  E = floor(log2 a) = ex - 1
    _, ex = np.frexp(a_fin)
    E = ex.astype(np.int64) - 1
    q = np.rint(np.ldexp(a_fin, -(E - 3))).astype(np.int64)    # in [8, 16]
    carry = q == 16
    E = np.where(carry, E + 1, E)
    q = np.where(carry, 8, q)
    code_norm = ((E + 7) << 3) | (q - 8)

    code = np.where(a_fin < 2.0 ** -6, q_sub, code_norm)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = code | np.where(neg, 0x80, 0)
    code = np.where(nan, E4M3_NAN, code)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# Block quantisation along the last axis
# --------------------------------------------------------------------------
def quantize(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8-quantise ``x`` (fp64, last axis K, K % 32 == 0).

    Returns (x_q uint8 E4M3 codes, same shape; x_scale uint8 E8M0,
    ``[..., K // 32]`` row-major), the layout the aiter_flydsl page gives for
    activation scales and compressed_tensors_w8a8_mxfp8 gives for weights.

    Per block: amax = max |x_j| (exact in fp64), byte = :func:`scale_bytes`,
    element = E4M3_RNE_satfinite(x_j / 2**e), exact division by a power of
    two.  Blocks with a NaN or Inf get 0xFF and all elements 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    xb = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    amax = np.max(np.abs(xb), axis=-1)          # NaN propagates
    s = scale_bytes(amax)
    e = block_exponent(amax)
    v = np.ldexp(xb, -e[..., None])
    q = e4m3_encode(v)
    q = np.where((s == E8M0_NAN)[..., None], E4M3_NAN, q).astype(np.uint8)
    return q.reshape(x.shape), s


def dequantize(q: np.ndarray, s: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """Element value (E4M3, or an FP6 format) times 2**(byte - 127) per
    element, exact in fp64."""
    q = np.asarray(q)
    K = q.shape[-1]
    val = e4m3_value(q) if fmt == "e4m3" else fp6_value(q, fmt)
    v = val.reshape(*q.shape[:-1], K // BLOCK, BLOCK)
    return (v * e8m0_value(s)[..., None]).reshape(q.shape)


# --------------------------------------------------------------------------
# Linear layer
# --------------------------------------------------------------------------
def linear(x_q: np.ndarray, x_scale: np.ndarray, w_q: np.ndarray, w_scale: np.ndarray,
           bias: np.ndarray | None = None, w_format: str = "e4m3") -> np.ndarray:
    """out[m, n] = sum_k deq(x)[m, k] * deq(w)[n, k] + bias[n], in fp64.

    ``x_q`` is ``[M, K]`` (or ``[B, M, K]``) E4M3, ``w_q`` is ``[N, K]`` (or
    ``[B, N, K]``) with elements in ``w_format`` ("e4m3", or the MXFP6
    "e2m3" / "e3m2"), with row-major block scales.  The product over k is one
    fp64 matmul (a library step); nothing is rounded to bf16 here.  In the
    batched form each batch index uses its own activation and weight, and the
    bias (shape ``[N]``) is shared.
    """
    dx = dequantize(x_q, x_scale)
    dw = dequantize(w_q, w_scale, w_format)
    out = np.matmul(dx, np.swapaxes(dw, -1, -2))
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)
    return out


def linear_bf16(x: np.ndarray, w_q: np.ndarray, w_scale: np.ndarray,
                bias: np.ndarray | None = None) -> np.ndarray:
    """The dynamic path: quantise fp64 (bf16-valued) ``x``, then :func:`linear`."""
    x_q, x_s = quantize(x)
    return linear(x_q, x_s, w_q, w_scale, bias)


# --------------------------------------------------------------------------
# MXFP6 weight elements (OCP MX v1.0, section 5.3.2: FP6 E2M3 and E3M2)
# --------------------------------------------------------------------------
# Both have no infinities and no NaN; a code is S.E...E.M...M in the low 6
# bits of a byte.  E2M3: 2 exponent bits, bias 1, 3 mantissa bits, largest
# finite 1.875 * 2**2 = 7.5.  E3M2: 3 exponent bits, bias 3, 2 mantissa bits,
# largest finite 1.75 * 2**4 = 28.  The MX block exponent for these elements
# is floor(log2 amax) - emax with emax = 2 (E2M3) or 4 (E3M2), so a block's
# largest element lands in [2**emax, 2**(emax+1)) before rounding, like the
# 8 of E4M3.
FP6_FORMATS = {"e2m3": (2, 3, 1), "e3m2": (3, 2, 3)}   # exponent bits, mantissa bits, bias


def fp6_emax(fmt: str) -> int:
    """Exponent of the largest normal binade: (2**ebits - 1) - bias."""
    ebits, _, bias = FP6_FORMATS[fmt]
    return (2 ** ebits - 1) - bias


def fp6_max(fmt: str) -> float:
    """Largest finite magnitude, (2 - 2**-mbits) * 2**emax."""
    _, mbits, _ = FP6_FORMATS[fmt]
    return (2.0 - 2.0 ** -mbits) * 2.0 ** fp6_emax(fmt)


def fp6_value(code: np.ndarray, fmt: str) -> np.ndarray:
    """Value of an FP6 code: normal (2**mbits + m) * 2**(e - bias - mbits),
    subnormal (e = 0) m * 2**(1 - bias - mbits)."""
    ebits, mbits, bias = FP6_FORMATS[fmt]
    c = np.asarray(code).astype(np.int64) & 0x3F
    s = np.where(c & 0x20, -1.0, 1.0)
    e = (c >> mbits) & ((1 << ebits) - 1)
    m = c & ((1 << mbits) - 1)
    normal = np.ldexp(((1 << mbits) + m).astype(np.float64), e - bias - mbits)
    sub = np.ldexp(m.astype(np.float64), 1 - bias - mbits)
    return s * np.where(e == 0, sub, normal)


def fp6_encode(v: np.ndarray, fmt: str) -> np.ndarray:
    """Round fp64 values to FP6 codes: nearest, ties to even, saturating.

    |v| >= the largest finite value (Inf included) gives the largest code
    (0x1F, with the sign); NaN gives 0x00 (FP6 has no NaN: a block holding
    one is marked NaN by its scale byte instead).  Below the smallest normal
    2**(1 - bias) the grid is the subnormal one, step 2**(1 - bias - mbits);
    from 2**E up to 2**(E+1) the step is 2**(E - mbits).  The sign is kept, so
    a value that rounds to zero gives 0x00 or 0x20.
    """
    ebits, mbits, bias = FP6_FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(v)
    top = fp6_max(fmt)
    a_fin = np.where(nan | (a >= top), 0.0, a)

    # subnormal range: q steps of 2**(1 - bias - mbits); q == 2**mbits is the smallest normal
    q_sub = np.rint(np.ldexp(a_fin, bias + mbits - 1)).astype(np.int64)

    # normal range: E = floor(log2 a), q = a / 2**(E - mbits) in [2**mbits, 2**(mbits+1)]
    _, ex = np.frexp(a_fin)
    E = ex.astype(np.int64) - 1
    q = np.rint(np.ldexp(a_fin, -(E - mbits))).astype(np.int64)
    carry = q == (2 << mbits)
    E = np.where(carry, E + 1, E)
    q = np.where(carry, 1 << mbits, q)
    code_norm = ((E + bias) << mbits) | (q - (1 << mbits))

    code = np.where(a_fin < 2.0 ** (1 - bias), q_sub, code_norm)
    code = np.where(a >= top, 0x1F, code)
    code = code | np.where(neg, 0x20, 0)
    code = np.where(nan, 0, code)
    return code.astype(np.uint8)


def quantize_fp6(x: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """MXFP6-quantise ``x`` (fp64, last axis K, K % 32 == 0) to ``fmt``.

    As :func:`quantize` with the FP6 element: per block amax, byte =
    :func:`scale_bytes` with emax of ``fmt``, element =
    FP6_RNE_satfinite(x_j / 2**e).  Returns (codes uint8, one 6-bit code per
    byte, same shape; scales uint8 ``[..., K // 32]``).  A block with a NaN or
    Inf gets scale 0xFF and all codes 0x00.
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    emax = fp6_emax(fmt)
    xb = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    amax = np.max(np.abs(xb), axis=-1)          # NaN propagates
    s = scale_bytes(amax, emax)
    e = block_exponent(amax, emax)
    q = fp6_encode(np.ldexp(xb, -e[..., None]), fmt)
    q = np.where((s == E8M0_NAN)[..., None], 0, q).astype(np.uint8)
    return q.reshape(x.shape), s
