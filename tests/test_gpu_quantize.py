"""mxfp8_quantize on the GPU against the oracle: bit for bit, x_q and x_scale."""

import numpy as np
import pytest
import torch

import oracle
from _helpers import bf16_to_dev, device
from mxfp8_block_scaled_02_gb300 import ops, synth
from test_oracle import GOLDEN_BLOCKS

pytestmark = pytest.mark.gpu


def _gpu_quantize(bits: np.ndarray):
    dev = device()
    q, s = ops.quantize(bf16_to_dev(bits, dev))
    ops.check()
    return q.cpu().numpy(), s.cpu().numpy()


def _assert_exact(bits: np.ndarray):
    q, s = _gpu_quantize(bits)
    rq, rs = oracle.quantize(synth.bf16_bits_to_f64(bits))
    assert np.array_equal(s, rs), f"{int((s != rs).sum())} scale bytes differ"
    if not np.array_equal(q, rq):
        bad = np.argwhere(q != rq)[:5]
        raise AssertionError(f"{int((q != rq).sum())} codes differ, first at {bad.tolist()}: "
                             f"gpu {[hex(q[tuple(i)]) for i in bad]} oracle {[hex(rq[tuple(i)]) for i in bad]}")


def test_hand_worked_blocks_on_gpu():
    x = np.stack([b["x"] for b in GOLDEN_BLOCKS])
    bits = synth.to_bf16_bits(x)
    q, s = _gpu_quantize(bits)
    for i, b in enumerate(GOLDEN_BLOCKS):
        assert int(s[i, 0]) == b["scale"], (b["name"], hex(s[i, 0]))
        assert np.array_equal(q[i], b["q"]), (b["name"], [hex(v) for v in q[i]])


def test_every_bf16_pattern():
    """All 65536 bf16 bit patterns, in order and in a fixed shuffle, as 32-blocks."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    _assert_exact(allbits.reshape(-1, 1024))
    perm = (np.arange(65536, dtype=np.int64) * 40503) % 65536
    _assert_exact(allbits[perm].reshape(-1, 2048))


def test_e4m3_rounding_grid_at_unit_scale():
    """Blocks led by 448 (scale 2^0), filled with every bf16 value in [-448, 448]."""
    b = np.arange(0, 0x43E1, dtype=np.uint16)          # 0 .. 448 in bf16 bits
    v = np.concatenate([b, b | np.uint16(0x8000)])
    pad = (-v.size) % 31
    v = np.concatenate([v, np.zeros(pad, np.uint16)]).reshape(-1, 31)
    lead = np.full((v.shape[0], 1), 0x43E0, np.uint16)   # 448.0
    _assert_exact(np.concatenate([lead, v], axis=1))


@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (7, 512), (129, 4096), (5, 14336)])
def test_ragged_shapes(rows, K):
    p = synth.make_problem("r", 1, rows, 8, K, seed=rows * 7 + K, outlier_frac=1e-2,
                           zero_block_frac=5e-2)
    _assert_exact(p.x[0])


@pytest.mark.parametrize("name", ["tiny", "decode64", "prefill_up"])
def test_workload_activations(name):
    p = synth.WORKLOADS[name]()
    _assert_exact(p.x.reshape(-1, p.K))


def test_bmm_activations():
    p = synth.bmm()
    _assert_exact(p.x.reshape(-1, p.K))


def test_quantize_scale_extremes():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)) * np.ldexp(1.0, rng.integers(-140, 126, (64, 1)))
    _assert_exact(synth.to_bf16_bits(x))


def test_zero_rows_is_noop():
    dev = device()
    q, s = ops.quantize(torch.empty((0, 64), dtype=torch.bfloat16, device=dev))
    ops.check()
    assert q.shape == (0, 64) and s.shape == (0, 2)
