"""Shared helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""

import numpy as np
import pytest
import torch

import oracle
from mxfp8_block_scaled_02_gb300 import build, ops, synth

_built = False


def device() -> torch.device:
    global _built
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not _built:
        build.build()
        ops.load()
        _built = True
    return torch.device("cuda:0")


def bf16_to_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8_to_dev(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def oracle_weights(p: synth.LinearProblem):
    """E4M3 weights and row-major scales from the oracle quantiser, [B, N, K]."""
    return oracle.quantize(synth.bf16_bits_to_f64(p.w))


def tolerance_violations(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    return ~(np.abs(out - ref) <= 1e-2 * (np.abs(ref) + 1e-2 * rms))


def assert_close(out_bf16: torch.Tensor, ref: np.ndarray, what: str = "") -> None:
    got = out_bf16.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bad = tolerance_violations(got, ref)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        detail = ", ".join(f"{tuple(i)}: got {got[tuple(i)]:.6g} ref {ref[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; {detail}")
