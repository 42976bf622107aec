"""Thin ctypes binding over libmxfp8.so (include/mxfp8.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  There is no
fallback: if the library is missing or the GPU is not sm_103, calls raise.

Shapes follow the vLLM pages: "CompressedTensorsW8A8Mxfp8.create_weights"
(weight [N, K] E4M3, weight_scale [N, K // 32] uint8) and
"AiterFlyDSLMxfp8LinearKernel.apply_weights" (x [..., K] bf16 or a
pre-quantised x_q [..., K] with row-major scales [..., K // 32]; output
[..., N] in bf16, plus bias).
"""

from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxfp8.so")
BLOCK = 32

_STATUS = {0: "MXFP8_OK", 1: "MXFP8_ERR_INVALID_ARG", 2: "MXFP8_ERR_UNSUPPORTED",
           3: "MXFP8_ERR_ARCH", 4: "MXFP8_ERR_CUDA", 5: "MXFP8_ERR_TIMEOUT"}

# name -> (restype, argtypes), mirroring include/mxfp8.h
_P, _I64, _U64, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
_SIZE_P = ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "mxfp8_last_error": (ctypes.c_char_p, []),
    "mxfp8_version": (_INT, []),
    "mxfp8_quantize": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "mxfp8_packed_sizes": (_INT, [_I64, _I64, _I64, _SIZE_P, _SIZE_P]),
    "mxfp8_process_weights": (_INT, [_P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "mxfp8_unpack_scales": (_INT, [_P, _I64, _I64, _I64, _P, _P]),
    "mxfp8_workspace_size": (_INT, [_I64, _I64, _I64, _I64, _INT, _SIZE_P]),
    "mxfp8_linear": (_INT, [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P,
                            ctypes.c_size_t, _P]),
    "mxfp8_linear_path": (_INT, [_INT, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                 _P, ctypes.c_size_t, _P]),
    "mxfp8_quantize_packed": (_INT, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "mxfp8_pack_scales": (_INT, [_P, _I64, _I64, _I64, _P, _P]),
    "mxfp8_gemm_packed": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "mxfp8_linear_noalloc": (_INT, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "mxfp8_linear_quantized_out": (_INT, [_P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P,
                                          _P, ctypes.c_size_t, _P]),
    "mxfp8_gemm_packed_quantized_out": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P,
                                               _P]),
    "mxfp8_blob_size": (_INT, [_I64, _I64, _I64, _INT, _SIZE_P]),
    "mxfp8_weights_serialize": (_INT, [_P, _P, _I64, _I64, _I64, _INT, _INT, _P, ctypes.c_size_t]),
    "mxfp8_weights_deserialize": (_INT, [_P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                         _SIZE_P, _SIZE_P]),
    "mxfp8_quantize_weights": (_INT, [_P, _I64, _I64, _INT, _P, _P, _P]),
    "mxfp8_packed_sizes_fmt": (_INT, [_INT, _I64, _I64, _I64, _SIZE_P, _SIZE_P]),
    "mxfp8_process_weights_fmt": (_INT, [_INT, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
    "mxfp8_linear_fmt": (_INT, [_INT, _INT, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P,
                                ctypes.c_size_t, _P]),
    "mxfp8_check": (_INT, [_P]),
    "mxfp8_debug_expire_wait": (_INT, [_U64, _P]),
}

_lib = None

# weight element formats (MXFP8_WFMT_*): E4M3 (MXFP8) and the MXFP6 E2M3 / E3M2
WFMT = {"e4m3": 0, "e2m3": 1, "e3m2": 2}


class MxStatusError(RuntimeError):
    def __init__(self, status: int, text: str):
        self.status = status
        super().__init__(f"{_STATUS.get(status, status)}: {text}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmxfp8.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m mxfp8_block_scaled_02_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise MxStatusError(status, load().mxfp8_last_error().decode())


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _bytes(t: torch.Tensor) -> torch.Tensor:
    """Same memory viewed as uint8 (E4M3 / E8M0 tensors are passed as bytes)."""
    return t if t.dtype == torch.uint8 else t.view(torch.uint8)


def _require_cuda(*ts: torch.Tensor | None) -> None:
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensors must be on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


def _aligned16(t: torch.Tensor | None) -> torch.Tensor | None:
    """The same values at a 16-byte aligned address (every pointer the ABI takes
    must be; a view into a larger tensor may not be), copied only if needed."""
    if t is None or t.data_ptr() % 16 == 0:
        return t
    return t.clone(memory_format=torch.contiguous_format)


def quantize(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 x [..., K] -> (x_q uint8 E4M3 [..., K], x_scale uint8 E8M0 [..., K/32])."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    _require_cuda(x)
    x = _aligned16(x)
    K = x.shape[-1]
    rows = x.numel() // K if K else 0
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty((*x.shape[:-1], K // BLOCK), dtype=torch.uint8, device=x.device)
    _check(load().mxfp8_quantize(_ptr(x), rows, K, _ptr(q), _ptr(s), _stream()))
    return q, s


def packed_sizes(B: int, N: int, K: int, fmt: str = "e4m3") -> tuple[int, int]:
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mxfp8_packed_sizes_fmt(WFMT[fmt], B, N, K, ctypes.byref(wb), ctypes.byref(sb)))
    return wb.value, sb.value


def quantize_weights(w: torch.Tensor, fmt: str = "e4m3") -> tuple[torch.Tensor, torch.Tensor]:
    """bf16 weights [..., K] -> (codes uint8 [..., K], one per byte; scales uint8
    [..., K/32]) in ``fmt`` ("e4m3", or the MXFP6 "e2m3" / "e3m2")."""
    if w.dtype != torch.bfloat16:
        raise TypeError("w must be bfloat16")
    _require_cuda(w)
    w = _aligned16(w)
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    s = torch.empty((*w.shape[:-1], K // BLOCK), dtype=torch.uint8, device=w.device)
    _check(load().mxfp8_quantize_weights(_ptr(w), rows, K, WFMT[fmt], _ptr(q), _ptr(s), _stream()))
    return q, s


@dataclasses.dataclass
class PackedWeights:
    """Weights after the one-time repack: E4M3 bytes and scale atoms."""

    w_packed: torch.Tensor   # uint8, B*N*K bytes (3BNK/4 for packed FP6)
    sf_packed: torch.Tensor  # uint8, packed scale atoms
    B: int
    N: int
    K: int
    batched: bool
    fmt: str = "e4m3"        # weight element format: "e4m3", "e2m3" or "e3m2"


def process_weights(w_q: torch.Tensor, w_scale: torch.Tensor, fmt: str = "e4m3") -> PackedWeights:
    """w_q [N, K] or [B, N, K] (uint8 or float8_e4m3fn; for ``fmt`` "e2m3" /
    "e3m2" one FP6 code per byte), w_scale [..., K/32] uint8.

    A checkpoint may store its scales padded (more rows than N or more blocks
    than K/32, as the aiter_flydsl page's process_weights_after_loading slices
    them with ``[:N, :K // 32]``): the padding is sliced off here and the
    scales copied to a dense, aligned tensor before the repack.
    """
    if w_q.dim() not in (2, 3):
        raise ValueError("w_q must be [N, K] or [B, N, K]")
    batched = w_q.dim() == 3
    B = w_q.shape[0] if batched else 1
    N, K = w_q.shape[-2], w_q.shape[-1]
    if K % BLOCK:
        raise ValueError(f"K={K} is not a multiple of {BLOCK}")
    if (w_scale.dim() != w_q.dim() or tuple(w_scale.shape[:-2]) != tuple(w_q.shape[:-2])
            or w_scale.shape[-2] < N or w_scale.shape[-1] < K // BLOCK):
        raise ValueError(f"weight scale {tuple(w_scale.shape)} does not match weight {tuple(w_q.shape)}")
    w_scale = w_scale[..., :N, :K // BLOCK]
    if not w_scale.is_contiguous():
        w_scale = w_scale.contiguous()
    w_q, w_scale = _aligned16(w_q), _aligned16(w_scale)
    _require_cuda(w_q, w_scale)
    wb, sb = packed_sizes(B, N, K, fmt)
    wp = torch.empty(wb, dtype=torch.uint8, device=w_q.device)
    sp = torch.empty(sb, dtype=torch.uint8, device=w_q.device)
    _check(load().mxfp8_process_weights_fmt(WFMT[fmt], _ptr(_bytes(w_q)), _ptr(_bytes(w_scale)), B, N, K,
                                            _ptr(wp), _ptr(sp), _stream()))
    return PackedWeights(wp, sp, B, N, K, batched, fmt)


def save_packed(pw: PackedWeights) -> bytes:
    """The packed weights as one self-describing blob (mxfp8_weights_serialize):
    a versioned, checksummed header, then the w_packed and sf_packed bytes.
    Write it to a file once; load_packed restores it without repacking."""
    w = np.ascontiguousarray(pw.w_packed.detach().cpu().numpy())
    sf = np.ascontiguousarray(pw.sf_packed.detach().cpu().numpy())
    n = ctypes.c_size_t()
    _check(load().mxfp8_blob_size(pw.B, pw.N, pw.K, WFMT[pw.fmt], ctypes.byref(n)))
    if (w.size, sf.size) != packed_sizes(pw.B, pw.N, pw.K, pw.fmt):
        raise ValueError("packed tensors do not have the sizes of (B, N, K)")
    blob = np.empty(n.value, dtype=np.uint8)
    _check(load().mxfp8_weights_serialize(w.ctypes.data, sf.ctypes.data, pw.B, pw.N, pw.K, WFMT[pw.fmt],
                                          int(pw.batched), blob.ctypes.data, blob.size))
    return blob.tobytes()


def load_packed(blob: bytes | bytearray | memoryview, device: torch.device | str) -> PackedWeights:
    """PackedWeights from a blob written by save_packed (checked by
    mxfp8_weights_deserialize: format, layout, sizes and both checksums),
    copied to ``device``."""
    buf = np.frombuffer(blob, dtype=np.uint8)
    B, N, K = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    fmt, batched = ctypes.c_int(), ctypes.c_int()
    wo, so = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mxfp8_weights_deserialize(buf.ctypes.data, buf.size, ctypes.byref(B), ctypes.byref(N),
                                            ctypes.byref(K), ctypes.byref(fmt), ctypes.byref(batched),
                                            ctypes.byref(wo), ctypes.byref(so)))
    name = {v: k for k, v in WFMT.items()}[fmt.value]
    wb, sb = packed_sizes(B.value, N.value, K.value, name)
    w = torch.from_numpy(buf[wo.value:wo.value + wb].copy()).to(device)
    sf = torch.from_numpy(buf[so.value:so.value + sb].copy()).to(device)
    return PackedWeights(w, sf, B.value, N.value, K.value, bool(batched.value), name)


def unpack_scales(pw: PackedWeights) -> torch.Tensor:
    out = torch.empty((pw.B, pw.N, pw.K // BLOCK), dtype=torch.uint8, device=pw.sf_packed.device)
    _check(load().mxfp8_unpack_scales(_ptr(pw.sf_packed), pw.B, pw.N, pw.K, _ptr(out), _stream()))
    return out if pw.batched else out[0]


def workspace_size(B: int, M: int, N: int, K: int, quantized: bool) -> int:
    n = ctypes.c_size_t()
    _check(load().mxfp8_workspace_size(B, M, N, K, int(quantized), ctypes.byref(n)))
    return n.value


def _linear_rows(x: torch.Tensor, pw: PackedWeights, bias: torch.Tensor | None,
                 x_scale: torch.Tensor | None, out: torch.Tensor | None) -> int:
    """Check x (and x_scale, bias, out) against the packed weights; returns M,
    the rows per batch.  Shared by every linear entry point, so that none of
    them hands the library a buffer shorter than the sizes it is told."""
    quantized = x_scale is not None
    if not quantized and x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16 (or pass x_scale with a pre-quantised x)")
    if quantized and x.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError("a pre-quantised x must be uint8 or float8_e4m3fn E4M3 codes")
    _require_cuda(x, x_scale, bias, out)
    if x.dim() < 1:
        raise ValueError("x must have a K dimension")
    K = x.shape[-1]
    if K != pw.K:
        raise ValueError(f"x has K={K}, weights have K={pw.K}")
    if pw.batched:
        if x.dim() != 3 or x.shape[0] != pw.B:
            raise ValueError("batched weights need x of shape [B, M, K]")
        M = x.shape[1]
    else:
        M = x.numel() // K if K else 0
    if quantized and (x_scale.dtype not in (torch.uint8, torch.float8_e8m0fnu)
                      or tuple(x_scale.shape) != (*x.shape[:-1], K // BLOCK)):
        raise ValueError(f"MXFP8 activation scale {tuple(x_scale.shape)} for {tuple(x.shape)}")
    if bias is not None and (bias.dtype != torch.bfloat16 or tuple(bias.shape) != (pw.N,)):
        raise ValueError("bias must be bf16 [N]")
    if out is not None and (out.dtype != torch.bfloat16 or out.numel() != pw.B * M * pw.N):
        raise ValueError(f"out must be bf16 with {pw.B * M * pw.N} elements")
    return M


def linear(x: torch.Tensor, pw: PackedWeights, bias: torch.Tensor | None = None,
           x_scale: torch.Tensor | None = None, *, path: int = 0,
           out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """MXFP8 linear layer.

    ``x`` is bf16 ``[..., K]`` (quantised inside the call), or with ``x_scale``
    given, the pre-quantised E4M3 ``x_q [..., K]`` with row-major scales
    ``[..., K/32]``.  For batched weights (``[B, N, K]``) x is ``[B, M, K]``.
    Returns bf16 ``[..., N]``.  ``path`` forces the small-M (1) or large-M (2)
    kernel path, the large-M path on CTA-pair tiles (3), the large-M kernels
    without the small-M one (4), or the GEMM that quantises bf16 x itself (5);
    0 lets the library choose.
    """
    quantized = x_scale is not None
    M = _linear_rows(x, pw, bias, x_scale, out)
    K = pw.K
    x, x_scale, bias = _aligned16(x), _aligned16(x_scale), _aligned16(bias)
    if out is None:
        out = torch.empty((*x.shape[:-1], pw.N), dtype=torch.bfloat16, device=x.device)
    if M == 0:
        return out
    ws_bytes = workspace_size(pw.B, M, pw.N, K, quantized)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=x.device)
    xb = None if quantized else x
    xq = _bytes(x) if quantized else None
    _check(load().mxfp8_linear_fmt(path, WFMT[pw.fmt], _ptr(xb), _ptr(xq), _ptr(x_scale), pw.B, M, pw.N, K,
                                   _ptr(pw.w_packed), _ptr(pw.sf_packed), _ptr(bias), _ptr(out),
                                   _ptr(workspace), workspace.numel(), _stream()))
    return out


def _e4m3_only(pw: PackedWeights, what: str) -> None:
    if pw.fmt != "e4m3":
        raise ValueError(f"{what} takes E4M3 weights only (these are {pw.fmt}); use linear")


@dataclasses.dataclass
class PackedActivation:
    """Activations quantised straight into the GEMM's operand layout."""

    x_q: torch.Tensor        # uint8 [B, M, K]
    sf_packed: torch.Tensor  # uint8 packed scale atoms
    B: int
    M: int
    K: int


def quantize_packed(x: torch.Tensor, B: int = 1, *, x_q: torch.Tensor | None = None,
                    sf_packed: torch.Tensor | None = None) -> PackedActivation:
    """bf16 x ([M, K], or [B, M, K] with B given) -> E4M3 codes + packed scales."""
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    _require_cuda(x)
    x = _aligned16(x)
    K = x.shape[-1]
    M = x.numel() // (K * B)
    if x_q is None:
        x_q = torch.empty((B, M, K), dtype=torch.uint8, device=x.device)
    if sf_packed is None:
        sf_packed = torch.empty(packed_sizes(B, max(M, 1), K)[1], dtype=torch.uint8, device=x.device)
    _check(load().mxfp8_quantize_packed(_ptr(x), B, M, K, _ptr(x_q), _ptr(sf_packed), _stream()))
    return PackedActivation(x_q, sf_packed, B, M, K)


def pack_scales(scale: torch.Tensor, B: int = 1) -> torch.Tensor:
    """Row-major E8M0 scales [B, R, K/32] (or [R, K/32]) -> packed atoms."""
    _require_cuda(scale)
    scale = _aligned16(scale)
    KB = scale.shape[-1]
    R = scale.numel() // (KB * B)
    out = torch.empty(packed_sizes(B, R, KB * BLOCK)[1], dtype=torch.uint8, device=scale.device)
    _check(load().mxfp8_pack_scales(_ptr(_bytes(scale)), B, R, KB * BLOCK, _ptr(out), _stream()))
    return out


def gemm_packed(pa: PackedActivation, pw: PackedWeights, bias: torch.Tensor | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """The block-scaled GEMM + bias epilogue alone; returns bf16 [B, M, N]."""
    _e4m3_only(pw, "gemm_packed")
    if pa.K != pw.K or pa.B != pw.B:
        raise ValueError("activation and weights disagree on K or B")
    _require_cuda(bias, out)
    if out is not None and (out.dtype != torch.bfloat16 or out.numel() != pa.B * pa.M * pw.N):
        raise ValueError(f"out must be bf16 with {pa.B * pa.M * pw.N} elements")
    if out is None:
        out = torch.empty((pa.B, pa.M, pw.N), dtype=torch.bfloat16, device=pa.x_q.device)
    _check(load().mxfp8_gemm_packed(_ptr(pa.x_q), _ptr(pa.sf_packed), pa.B, pa.M, pw.N, pa.K,
                                    _ptr(pw.w_packed), _ptr(pw.sf_packed), _ptr(bias), _ptr(out),
                                    _stream()))
    return out


def _hand_off_buffers(B: int, M: int, N: int, device) -> PackedActivation:
    y_q = torch.empty((B, M, N), dtype=torch.uint8, device=device)
    y_sf = torch.empty(packed_sizes(B, max(M, 1), N)[1], dtype=torch.uint8, device=device)
    return PackedActivation(y_q, y_sf, B, M, N)


def linear_quantized_out(x: torch.Tensor, pw: PackedWeights, bias: torch.Tensor | None = None,
                         x_scale: torch.Tensor | None = None, *, bf16_out: bool = True,
                         workspace: torch.Tensor | None = None
                         ) -> tuple[torch.Tensor | None, PackedActivation]:
    """MXFP8 linear layer that also hands its output on quantised
    (mxfp8_linear_quantized_out): returns (bf16 out or None, y as a
    PackedActivation that gemm_packed / gemm_packed_quantized_out take as x)."""
    _e4m3_only(pw, "linear_quantized_out")
    M = _linear_rows(x, pw, bias, x_scale, None)
    quantized = x_scale is not None
    x, x_scale, bias = _aligned16(x), _aligned16(x_scale), _aligned16(bias)
    out = torch.empty((*x.shape[:-1], pw.N), dtype=torch.bfloat16, device=x.device) if bf16_out else None
    y = _hand_off_buffers(pw.B, M, pw.N, x.device)
    if M == 0:
        return out, y
    if workspace is None:
        workspace = torch.empty(max(workspace_size(pw.B, M, pw.N, pw.K, quantized), 1), dtype=torch.uint8,
                                device=x.device)
    xb = None if quantized else x
    xq = _bytes(x) if quantized else None
    _check(load().mxfp8_linear_quantized_out(_ptr(xb), _ptr(xq), _ptr(x_scale), pw.B, M, pw.N, pw.K,
                                             _ptr(pw.w_packed), _ptr(pw.sf_packed), _ptr(bias), _ptr(out),
                                             _ptr(y.x_q), _ptr(y.sf_packed), _ptr(workspace),
                                             workspace.numel(), _stream()))
    return out, y


def gemm_packed_quantized_out(pa: PackedActivation, pw: PackedWeights, bias: torch.Tensor | None = None,
                              *, bf16_out: bool = True) -> tuple[torch.Tensor | None, PackedActivation]:
    """gemm_packed whose output is also handed on quantised
    (mxfp8_gemm_packed_quantized_out): the middle layer of a chain."""
    _e4m3_only(pw, "gemm_packed_quantized_out")
    if pa.K != pw.K or pa.B != pw.B:
        raise ValueError("activation and weights disagree on K or B")
    _require_cuda(bias)
    out = torch.empty((pa.B, pa.M, pw.N), dtype=torch.bfloat16, device=pa.x_q.device) if bf16_out else None
    y = _hand_off_buffers(pa.B, pa.M, pw.N, pa.x_q.device)
    _check(load().mxfp8_gemm_packed_quantized_out(_ptr(pa.x_q), _ptr(pa.sf_packed), pa.B, pa.M, pw.N, pa.K,
                                                  _ptr(pw.w_packed), _ptr(pw.sf_packed), _ptr(bias), _ptr(out),
                                                  _ptr(y.x_q), _ptr(y.sf_packed), _stream()))
    return out, y


NOALLOC_SCRATCH_BYTES = 32 << 20


def linear_noalloc(x: torch.Tensor, pw: PackedWeights, bias: torch.Tensor | None = None,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 linear that allocates no device workspace (mxfp8_linear_noalloc).

    For callers that cannot allocate device memory: the library's fixed
    32 MiB scratch array holds the quantised activations, so B*M*K is limited
    (the call raises MXFP8_ERR_UNSUPPORTED beyond it).  Calls that overlap on
    the GPU share that array and race.  Only ``out`` is allocated here when it
    is not given.
    """
    _e4m3_only(pw, "linear_noalloc")
    M = _linear_rows(x, pw, bias, None, out)
    K = pw.K
    x, bias = _aligned16(x), _aligned16(bias)
    if out is None:
        out = torch.empty((*x.shape[:-1], pw.N), dtype=torch.bfloat16, device=x.device)
    if M == 0:
        return out
    _check(load().mxfp8_linear_noalloc(_ptr(x), pw.B, M, pw.N, K, _ptr(pw.w_packed),
                                       _ptr(pw.sf_packed), _ptr(bias), _ptr(out), _stream()))
    return out


def check() -> None:
    """Synchronise the current stream and raise if a kernel wait ran out."""
    _check(load().mxfp8_check(_stream()))


def debug_expire_wait(timeout_ns: int) -> None:
    _check(load().mxfp8_debug_expire_wait(timeout_ns, _stream()))
