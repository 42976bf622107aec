"""Packed weights restored from a blob give the same layer output bit for bit
as the weights they were saved from (the pre-processed weights are used as
they are, with no repack)."""

import numpy as np
import pytest
import torch

from _helpers import bf16_to_dev, device, oracle_weights, u8_to_dev
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,M,N,K", [(1, 16, 4096, 4096), (1, 300, 520, 1024), (3, 200, 264, 256)])
def test_restored_weights_give_identical_output(B, M, N, K, tmp_path):
    dev = device()
    p = synth.make_problem("blob", B, M, N, K, seed=90 + M, bias_std=0.1)
    wq, ws = oracle_weights(p)
    batched = B > 1
    pw = ops.process_weights(u8_to_dev(wq if batched else wq[0], dev), u8_to_dev(ws if batched else ws[0], dev))
    path = tmp_path / "w.mxfp8"
    path.write_bytes(ops.save_packed(pw))
    back = ops.load_packed(path.read_bytes(), dev)
    assert (back.B, back.N, back.K, back.batched) == (pw.B, pw.N, pw.K, pw.batched)
    assert torch.equal(back.w_packed, pw.w_packed) and torch.equal(back.sf_packed, pw.sf_packed)

    x = bf16_to_dev(p.x if batched else p.x[0], dev)
    bias = bf16_to_dev(p.bias, dev)
    a = ops.linear(x, pw, bias)
    b = ops.linear(x, back, bias)
    ops.check()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert np.isfinite(a.float().cpu().numpy()).all()
