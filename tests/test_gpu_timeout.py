"""The bounded-wait path: a kernel whose wait can never complete returns on its
own, the status word reports MXFP8_ERR_TIMEOUT, and the context stays usable."""

import numpy as np
import pytest
import torch

from _helpers import bf16_to_dev, device
from mxfp8_block_scaled_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    dev = device()
    ops.check()                                   # clean state
    ops.debug_expire_wait(50_000_000)             # 50 ms
    with pytest.raises(ops.MxStatusError) as ei:
        ops.check()
    assert ei.value.status == 5
    ops.check()                                   # the status word was cleared
    # the device still runs the real kernels
    p = synth.make_problem("after", 1, 4, 64, 128, seed=2)
    q, s = ops.quantize(bf16_to_dev(p.x[0], dev))
    ops.check()
    torch.cuda.synchronize()
    assert q.shape == (4, 128) and np.isfinite(s.cpu().numpy()).all()
