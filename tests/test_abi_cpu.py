"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every symbol that
include/moe_nvfp4.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import nvfp4_mixture_experts_bf16_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ("moe_pack_nvfp4", "moe_route_topk", "moe_forward", "moe_quantize_act_nvfp4",
              "moe_workspace_size", "moe_pack_destroy", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    assert set(moe.EXPORTED) <= set(_declared())


def test_library_is_sm103a_only():
    # the build emits exactly one target, the architecture-specific sm_103a
    from nvfp4_mixture_experts_bf16_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(L):
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(5) == "MOE_ERR_TIMEOUT"
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_argument_validation_before_any_launch(L):
    vp = ctypes.c_void_p
    n = ctypes.c_size_t()
    # sizes
    assert L.moe_route_workspace_size(0, 512, 64, 4, ctypes.byref(n)) == 1      # T = 0
    assert L.moe_route_workspace_size(4, 500, 64, 4, ctypes.byref(n)) == 1      # H % 128
    assert L.moe_route_workspace_size(4, 512, 64, 65, ctypes.byref(n)) == 1     # k > E
    assert L.moe_route_workspace_size(4, 512, 64, 33, ctypes.byref(n)) == 1     # k > 32
    assert L.moe_route_workspace_size(4, 512, 2048, 4, ctypes.byref(n)) == 1    # E > 1024
    assert L.moe_route_workspace_size(4, 512, 64, 4, ctypes.byref(n)) == 0 and n.value > 0
    # null pointers / null pack
    assert L.moe_forward(None, None, None, 1, 1, 0, None, None, 0, None) == 1
    assert L.moe_workspace_size(None, 1, 1, 0, ctypes.byref(n)) == 1
    assert L.moe_quantize_act_nvfp4(None, 1, 16, ctypes.c_float(1.0), None, None, None) == 1
    # misaligned pointers are rejected (never dereferenced)
    assert L.moe_quantize_act_nvfp4(vp(8), 1, 16, ctypes.c_float(1.0), vp(16), vp(16), None) == 1
    # bad quantiser scale / shape
    assert L.moe_quantize_act_nvfp4(vp(16), 1, 16, ctypes.c_float(0.0), vp(16), vp(16), None) == 1
    assert L.moe_quantize_act_nvfp4(vp(16), 1, 15, ctypes.c_float(1.0), vp(16), vp(16), None) == 1
    # pack: bad sizes rejected before any copy
    M = moe._Matrix * 1
    g = M()
    assert L.moe_pack_nvfp4(g, g, g, 1, 100, 64, None, ctypes.byref(vp())) == 1
    assert L.moe_pack_nvfp4(g, g, g, 1, 128, 64, None, ctypes.byref(vp())) == 1  # null codes
    assert L.moe_pack_destroy(None) == 0
    assert L.moe_read_device_status(None, None, None) == 1
    # shared expert: a null pack or a null / invalid descriptor, before any launch
    sh = moe._SharedExpert(16, 16, 16, 384)
    assert L.moe_forward_shared(None, None, None, ctypes.byref(sh), 1, 1, 0, None, None, 0,
                                None) == 1
    assert L.moe_workspace_size_shared(None, 1, 1, 0, 384, ctypes.byref(n)) == 1
    o = ctypes.c_size_t()
    assert L.moe_workspace_offsets_shared(None, 1, 1, 0, 384, ctypes.byref(o), None, None) == 1


def test_workspace_size_grows_with_tokens(L):
    a = moe.moe_route_workspace_size(1, 4096, 512, 10)
    b = moe.moe_route_workspace_size(8192, 4096, 512, 10)
    assert b > a > 0


def test_fault_injection_arguments(L):
    assert L.moe_test_inject_faults(-2, 0.0, 0) == 1          # no such CTA
    assert L.moe_test_inject_faults(-1, -1.0, 0) == 1         # negative wait bound
    assert L.moe_test_inject_faults(-1, 11.0, 0) == 1         # above the 10 s cap
    assert L.moe_test_inject_faults(-1, 0.0, -1) == 1
    assert L.moe_test_inject_faults(-1, 0.0, 0) == 0          # everything off


def test_pack_allocation_failure_returns_oom(L):
    # an injected failure of moe_pack_nvfp4's device allocation: MOE_ERR_OOM, no pack, and the
    # following allocation is not affected by the spent injection
    import numpy as np
    E, H, I = 2, 128, 64
    codes = np.zeros(I * H // 2, np.uint8)
    scales = np.full(I * H // 16, 0x38, np.uint8)
    arr = (moe._Matrix * E)()
    for e in range(E):
        arr[e].codes = codes.ctypes.data
        arr[e].scales = scales.ctypes.data
        arr[e].multiplier = 1.0
        arr[e].input_scale = 1.0
    out = ctypes.c_void_p(12345)
    try:
        assert L.moe_test_inject_faults(-1, 0.0, 1) == 0
        assert L.moe_pack_nvfp4(arr, arr, arr, E, H, I, None, ctypes.byref(out)) == 3
        assert out.value is None
    finally:
        assert L.moe_test_inject_faults(-1, 0.0, 0) == 0
