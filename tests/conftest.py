import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")


def gemm_tolerance_violations(out: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Mask of entries outside |out - ref| <= 1e-2 * (|ref| + 1e-2 * rms(ref row)).

    ``ref`` is the oracle's fp64 result; ``out`` the bf16 output widened to
    fp64.  rms is taken over the last axis (n) for each leading index (b, m).
    A bf16 rounding of an fp32 sum is at most 2**-9 relative, so the bound
    leaves room for fp32 accumulation-order differences and the single bf16
    rounding, and the rms term covers entries that cancel to near zero.
    """
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = 1e-2 * (np.abs(ref) + 1e-2 * rms)
    return ~(np.abs(out - ref) <= bound)
