"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up after its time limit, records the timeout bit in the
status word and returns; the context stays usable afterwards."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_completes_or_times_out():
    import block_diffusion_speculative_02_gb300 as dfl
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfl.dflash.dflash_selftest_wait(True, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
    t0 = time.perf_counter()
    dfl.dflash.dflash_selftest_wait(False, ws)       # nothing arrives
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert dfl.dflash_read_status(ws) & dfl.dflash.STATUS_BITS["timeout"]
    assert 0.5 < waited < 30.0
    # the context is still usable: ordinary work and another completed wait
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
    ws.zero_()
    dfl.dflash.dflash_selftest_wait(True, ws)
    torch.cuda.synchronize()
    assert dfl.dflash_read_status(ws) == 0
