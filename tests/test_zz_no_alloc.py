"""The routing entry point for callers that cannot allocate device memory
(moe_route_topk_noalloc: runtimes whose allocator is frozen after start-up, embedders handed
only their input and output buffers). Its workspace is a fixed device array inside the library;
this test checks, through the C ABI, that two calls in a row give the results of moe_route_topk
with a caller-provided workspace, on the decode and the grouped routing paths, that the array's
status word reads back clean, and that shapes beyond the array are refused. It is collected last
so that a run stopping at the first failure has run every other test."""
import numpy as np
import pytest
import torch

import synth
import nvfp4_mixture_experts_bf16_gb300 as moe

pytestmark = pytest.mark.gpu


def _dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("T,H,E,k", [(1, 4096, 512, 10), (8, 4096, 512, 10), (37, 512, 96, 6),
                                     (300, 1024, 128, 8)])
def test_noalloc_routing_matches_workspace_routing(T, H, E, k):
    moe.build()
    x = _dev(synth.activations(9, 0, T, H, zipf=True))
    wr = _dev(synth.router_weight(9, 0, E, H, zipf=True))
    ref = moe.moe_route_topk(x, wr, k)
    for _ in range(2):   # the array keeps the last call's contents: two calls in a row
        got = moe.moe_route_topk_noalloc(x, wr, k)
        torch.cuda.synchronize()
        for name in ("idx", "counts", "offsets", "perm"):
            assert torch.equal(got[name], ref[name]), name
        # same kernels, same inputs: the weights agree to FP32 rounding (here: exactly)
        np.testing.assert_allclose(got["w"].cpu().numpy(), ref["w"].cpu().numpy(), rtol=1e-6,
                                   atol=0)
    # the fixed array's status word (kept across calls until read): no wait gave up
    assert moe.moe_read_device_status(None) == 0


def test_noalloc_routing_refuses_shapes_beyond_its_array():
    moe.build()
    T, H, E, k = 2048, 512, 1024, 8     # 8 MiB of logits alone: beyond the fixed 4 MiB
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_topk_noalloc(x, wr, k)
    assert e.value.code == 6   # MOE_ERR_WORKSPACE
