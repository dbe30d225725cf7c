"""Bounded waits: a kernel whose barrier is never released must give up after its
limit, record TPMLP_ERR_TIMEOUT in the device status word and leave the context
usable.  Nothing here faults, traps or hangs the GPU."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_times_out_and_context_survives(cuda_lib):
    tpmlp = cuda_lib
    assert tpmlp.device_status(reset=True) == 0
    t0 = time.time()
    tpmlp.wait_timeout_selftest(50_000_000)  # 50 ms limit
    rc = tpmlp.device_status(reset=True)
    elapsed = time.time() - t0
    assert rc == -6, rc  # TPMLP_ERR_TIMEOUT
    assert elapsed < 10.0
    assert tpmlp.device_status() == 0  # reset worked
    # the context still runs the block
    blk = tpmlp.MLPBlock(16, 2, 64, 256, 2, True, torch.bfloat16)
    x = [torch.randn(8, 2, 64, device="cuda").bfloat16() for _ in range(2)]
    w1 = torch.randn(256, 64, device="cuda").bfloat16() * 0.02
    w2 = torch.randn(64, 256, device="cuda").bfloat16() * 0.02
    out = blk.forward(x, w1, w2)
    torch.cuda.synchronize()
    assert tpmlp.device_status() == 0
    assert torch.isfinite(torch.cat(out["z"])).all()
