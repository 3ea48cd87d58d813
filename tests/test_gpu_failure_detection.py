"""Device-side failure detection without any GPU fault: a bounded wait that is made to
run out (a barrier nothing arrives at) is reported by fp8fg_sync_status as a timeout,
the status word is cleared, and the context stays usable for real work."""
import time

import pytest
import torch

from fp8_fine_grained_cast_b300 import _lib, inputs, ops

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    stream = torch.cuda.current_stream().cuda_stream
    ops.sync_status()                                   # clean start
    t0 = time.time()
    _lib.fp8fg_selftest_wait_timeout(stream)
    with pytest.raises(_lib.Fp8fgError) as ei:
        ops.sync_status()
    assert ei.value.code == _lib.FP8FG_ERR_TIMEOUT
    assert 0.5 < time.time() - t0 < 30.0
    ops.sync_status()                                   # cleared
    t = inputs.tiny(cuda_device)
    q, s = ops.quant_act_1x128(t.x)                     # the context still works
    c = ops.blockscaled_gemm(q, s, *ops.quant_w_128x128(t.w), ops.SB_BLOCK_128x128, torch.float32)
    ops.sync_status()
    assert torch.isfinite(c).all()
