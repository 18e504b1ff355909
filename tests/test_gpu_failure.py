"""Failure detection on the GPU without faulting it: the fused narrow-call kernel's CTAs wait
for each other's results with bounded waits. With the test-only fault injection one CTA
publishes no router logits and the wait bound is 1 ms, so every other CTA's wait runs out: the
call must still finish (quickly), record MOE_ERR_TIMEOUT in the workspace status word, and leave
the GPU usable: after the injection is switched off, a call on the re-zeroed workspace gives
the same output as a call on a fresh one."""
import time

import numpy as np
import pytest
import torch

import nvfp4_mixture_experts_bf16_gb300 as moe
from _gpu_fixtures import dev_bf16, host_u16, pack_from_experts, small_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.lib()
    yield
    moe.moe_test_inject_faults()     # never leave an injection on for later tests


@pytest.mark.parametrize("T,mode,skip", [(1, 0, 5), (8, 0, 0), (4, 1, 151), (2, 2, 77)])
def test_wait_timeout_is_reported_and_the_gpu_stays_usable(T, mode, skip):
    H, E, k, I = 512, 256, 4, 128
    x, wr, ex = small_layer(T, H, E, k, I, seed=700 + T, zipf=T > 1)
    pack = pack_from_experts(ex)
    xd, wd = dev_bf16(x), dev_bf16(wr)
    ws = moe.new_workspace(moe.moe_workspace_size(pack, T, k, mode))
    ref = host_u16(moe.moe_forward(xd, wd, pack, k, mode))     # a fresh workspace
    torch.cuda.synchronize()
    try:
        moe.moe_test_inject_faults(skip_logits_cta=skip, wait_limit_seconds=0.001)
        t0 = time.time()
        moe.moe_forward(xd, wd, pack, k, mode, ws=ws)
        assert moe.moe_last_launch_count() == 1     # the fused kernel ran
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        moe.moe_test_inject_faults()
    assert moe.moe_read_device_status(ws) == 5      # MOE_ERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    ws.zero_()
    got = host_u16(moe.moe_forward(xd, wd, pack, k, mode, ws=ws))
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    assert np.array_equal(got, ref)
    pack.close()
