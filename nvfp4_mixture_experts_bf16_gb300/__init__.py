"""GB300 (sm_103a) NVFP4 routed-expert MoE feed-forward: thin Python binding of the C ABI.

Every step of the path runs in the CUDA library ``_build/libmoe_nvfp4.so`` (see
``include/moe_nvfp4.h``); this module only marshals arguments: torch tensors become device
pointers, the current torch stream becomes the ``stream`` argument, and status codes become
exceptions. PyTorch provides device memory and streams and nothing else. There is no CPU
fallback: if the library is missing, every call raises.

Names follow the C ABI: ``moe_pack_nvfp4``, ``moe_route_topk``, ``moe_forward``,
``moe_quantize_act_nvfp4`` and the helpers around them.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

W4A16 = 0
W4A4 = 1

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_WORKSPACE"}

EXPORTED = ["moe_pack_nvfp4", "moe_pack_destroy", "moe_pack_info", "moe_pack_get_matrix",
            "moe_workspace_size", "moe_route_workspace_size", "moe_route_topk", "moe_forward",
            "moe_workspace_offsets", "moe_quantize_act_nvfp4", "moe_read_device_status",
            "moe_status_string", "moe_last_launch_count", "moe_profile_next_forward",
            "moe_route_topk_noalloc", "moe_workspace_size_shared", "moe_forward_shared",
            "moe_workspace_offsets_shared", "moe_profile_kernel_name",
            "moe_workspace_size_layers", "moe_workspace_offsets_layers", "moe_forward_layers",
            "moe_test_inject_faults"]


class MoeError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class _Matrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("multiplier", ctypes.c_float), ("input_scale", ctypes.c_float)]


class _SharedExpert(ctypes.Structure):
    _fields_ = [("gate_up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate", ctypes.c_void_p), ("inter", ctypes.c_int)]


class _WsOffsets(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("idx", "w", "counts", "offsets", "perm", "slot_of", "x_codes", "x_scales",
                 "h_bf16", "h_codes", "h_scales", "y")]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
            L = ctypes.CDLL(path)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.moe_pack_nvfp4.argtypes = [vp, vp, vp, i32, i32, i32, vp, ctypes.POINTER(vp)]
            L.moe_pack_destroy.argtypes = [vp]
            L.moe_pack_info.argtypes = [vp, vp, vp, vp, vp]
            L.moe_pack_get_matrix.argtypes = [vp, i32, i32, vp, vp, vp, vp]
            L.moe_workspace_size.argtypes = [vp, i32, i32, i32, ctypes.POINTER(sz)]
            L.moe_route_workspace_size.argtypes = [i32, i32, i32, i32, ctypes.POINTER(sz)]
            L.moe_route_topk.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
            L.moe_forward.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, sz, vp]
            L.moe_workspace_offsets.argtypes = [vp, i32, i32, i32, ctypes.POINTER(_WsOffsets)]
            L.moe_quantize_act_nvfp4.argtypes = [vp, i32, i32, ctypes.c_float, vp, vp, vp]
            L.moe_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
            L.moe_status_string.argtypes = [i32]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_last_launch_count.argtypes = []
            L.moe_profile_next_forward.argtypes = [vp, i32]
            L.moe_profile_kernel_name.argtypes = [i32]
            L.moe_test_inject_faults.argtypes = [i32, ctypes.c_double, i32]
            L.moe_workspace_size_layers.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
            L.moe_workspace_offsets_layers.argtypes = [vp, i32, i32, i32, i32, i32,
                                                       ctypes.POINTER(_WsOffsets)]
            L.moe_forward_layers.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, sz, vp]
            L.moe_route_topk_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            L.moe_workspace_size_shared.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
            L.moe_forward_shared.argtypes = [vp, vp, vp, ctypes.POINTER(_SharedExpert), i32, i32,
                                             i32, vp, vp, sz, vp]
            L.moe_workspace_offsets_shared.argtypes = [vp, i32, i32, i32, i32,
                                                       ctypes.POINTER(sz), ctypes.POINTER(sz),
                                                       ctypes.POINTER(sz)]
            for n in EXPORTED:
                if n not in ("moe_status_string", "moe_profile_kernel_name"):
                    getattr(L, n).restype = ctypes.c_int
            L.moe_profile_kernel_name.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _check(fn, code):
    if code != 0:
        raise MoeError(fn, code)


def _stream(stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _bits(t):
    """BF16 tensor -> its device pointer (the ABI takes BF16 bit patterns)."""
    import torch
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected a BF16 tensor, got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return _ptr(t)


class Pack:
    """A library-owned expert pack (moe_pack_nvfp4 ... moe_pack_destroy)."""

    def __init__(self, handle, E, H, I, device_bytes):
        self.handle, self.E, self.H, self.I, self.device_bytes = handle, E, H, I, device_bytes

    def close(self):
        if self.handle:
            _check("moe_pack_destroy", lib().moe_pack_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def get_matrix(self, expert: int, which: int):
        """(codes, scales, multiplier, input_scale) of one matrix in checkpoint layout (numpy)."""
        import numpy as np
        rows, cols = (self.H, self.I) if which == 2 else (self.I, self.H)
        codes = np.empty((rows, cols // 2), np.uint8)
        scales = np.empty((rows, cols // 16), np.uint8)
        m = ctypes.c_float()
        s = ctypes.c_float()
        _check("moe_pack_get_matrix", lib().moe_pack_get_matrix(
            self.handle, expert, which, codes.ctypes.data_as(ctypes.c_void_p),
            scales.ctypes.data_as(ctypes.c_void_p), ctypes.byref(m), ctypes.byref(s)))
        return codes, scales, m.value, s.value


def moe_pack_nvfp4(gate, up, down, hidden: int, inter: int, stream=None) -> Pack:
    """gate/up/down: lists (one entry per expert) of (codes, scales, multiplier, input_scale);
    codes/scales are torch tensors (CUDA or CPU) or numpy arrays in checkpoint layout."""
    E = len(gate)
    keep = []

    def mat_array(lst):
        arr = (_Matrix * E)()
        for e, (codes, scales, mult, ins) in enumerate(lst):
            for a in (codes, scales):
                keep.append(a)
            arr[e].codes = codes.data_ptr() if hasattr(codes, "data_ptr") else codes.ctypes.data
            arr[e].scales = scales.data_ptr() if hasattr(scales, "data_ptr") else scales.ctypes.data
            arr[e].multiplier = float(mult)
            arr[e].input_scale = float(ins)
        return arr

    g, u, d = mat_array(gate), mat_array(up), mat_array(down)
    h = ctypes.c_void_p()
    _check("moe_pack_nvfp4", lib().moe_pack_nvfp4(g, u, d, E, hidden, inter, _stream(stream),
                                                   ctypes.byref(h)))
    nbytes = ctypes.c_size_t()
    _check("moe_pack_info", lib().moe_pack_info(h, None, None, None, ctypes.byref(nbytes)))
    return Pack(h, E, hidden, inter, nbytes.value)


def moe_workspace_size(pack: Pack, T: int, k: int, mode: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size", lib().moe_workspace_size(pack.handle, T, k, mode, ctypes.byref(n)))
    return n.value


def moe_route_workspace_size(T: int, H: int, E: int, k: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_route_workspace_size", lib().moe_route_workspace_size(T, H, E, k, ctypes.byref(n)))
    return n.value


def moe_workspace_offsets(pack: Pack, T: int, k: int, mode: int) -> dict:
    o = _WsOffsets()
    _check("moe_workspace_offsets", lib().moe_workspace_offsets(pack.handle, T, k, mode,
                                                                ctypes.byref(o)))
    return {n: getattr(o, n) for n, _ in _WsOffsets._fields_}


def new_workspace(nbytes: int, device=None):
    """A zero-filled workspace (the ABI requires zeros before first use)."""
    import torch
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def moe_route_topk(x, router_w, k: int, ws=None, stream=None):
    """Returns dict(idx [T,k] int32, w [T,k] float32, counts [E], offsets [E+1], perm [T*k])."""
    import torch
    T, H = x.shape
    E = router_w.shape[0]
    dev = x.device
    if ws is None:
        ws = new_workspace(moe_route_workspace_size(T, H, E, k), dev)
    out = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
               w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(T * k, dtype=torch.int32, device=dev))
    _check("moe_route_topk", lib().moe_route_topk(
        _bits(x), _bits(router_w), T, H, E, k, _ptr(out["idx"]), _ptr(out["w"]),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_route_topk_noalloc(x, router_w, k: int, stream=None):
    """moe_route_topk with the library's fixed device workspace (no workspace argument): for
    callers that cannot allocate device memory. Calls that overlap on the GPU race."""
    import torch
    T, H = x.shape
    E = router_w.shape[0]
    dev = x.device
    out = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
               w=torch.empty((T, k), dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(T * k, dtype=torch.int32, device=dev))
    _check("moe_route_topk_noalloc", lib().moe_route_topk_noalloc(
        _bits(x), _bits(router_w), T, H, E, k, _ptr(out["idx"]), _ptr(out["w"]),
        _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]), _stream(stream)))
    return out


def moe_forward(x, router_w, pack: Pack, k: int, mode: int, out=None, ws=None, stream=None):
    """out [T,H] BF16 = the routed-expert MoE step of x [T,H] BF16 (all on the GPU)."""
    import torch
    T, H = x.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = new_workspace(moe_workspace_size(pack, T, k, mode), x.device)
    _check("moe_forward", lib().moe_forward(_bits(x), _bits(router_w), pack.handle, T, k, mode,
                                            _bits(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_workspace_size_layers(pack: Pack, layers: int, T: int, k: int, mode: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size_layers", lib().moe_workspace_size_layers(
        pack.handle, layers, T, k, mode, ctypes.byref(n)))
    return n.value


def moe_workspace_offsets_layers(pack: Pack, layers: int, T: int, k: int, mode: int,
                                 layer: int) -> dict:
    o = _WsOffsets()
    _check("moe_workspace_offsets_layers", lib().moe_workspace_offsets_layers(
        pack.handle, layers, T, k, mode, layer, ctypes.byref(o)))
    return {n: getattr(o, n) for n, _ in _WsOffsets._fields_}


def moe_forward_layers(x, router_ws, packs, k: int, mode: int, out=None, ws=None, stream=None):
    """The chained MoE step of len(packs) layers: x [T,H] BF16 is layer 0's input, layer l+1
    reads layer l's output; returns out [layers,T,H] BF16 (out[l] = layer l's output)."""
    import torch
    T, H = x.shape
    L = len(packs)
    assert len(router_ws) == L
    if out is None:
        out = torch.empty((L, T, H), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = new_workspace(moe_workspace_size_layers(packs[0], L, T, k, mode), x.device)
    rw = (ctypes.c_void_p * L)(*[_bits(w).value for w in router_ws])
    pk = (ctypes.c_void_p * L)(*[p.handle.value if isinstance(p.handle, ctypes.c_void_p)
                                 else p.handle for p in packs])
    _check("moe_forward_layers", lib().moe_forward_layers(
        _bits(x), rw, pk, L, T, k, mode, _bits(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_workspace_size_shared(pack: Pack, T: int, k: int, mode: int, shared_inter: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size_shared", lib().moe_workspace_size_shared(
        pack.handle, T, k, mode, shared_inter, ctypes.byref(n)))
    return n.value


def moe_workspace_offsets_shared(pack: Pack, T: int, k: int, mode: int,
                                 shared_inter: int) -> dict:
    h, sg, y = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check("moe_workspace_offsets_shared", lib().moe_workspace_offsets_shared(
        pack.handle, T, k, mode, shared_inter, ctypes.byref(h), ctypes.byref(sg), ctypes.byref(y)))
    return dict(h=h.value, sigma=sg.value, y=y.value)


def moe_forward_shared(x, router_w, pack: Pack, shared, k: int, mode: int, out=None, ws=None,
                       stream=None):
    """moe_forward plus the shared expert; ``shared`` = (gate_up [2*Is, H], down [H, Is],
    gate [H]) BF16 CUDA tensors."""
    import torch
    gate_up, down, gate = shared
    T, H = x.shape
    Is = gate_up.shape[0] // 2
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = new_workspace(moe_workspace_size_shared(pack, T, k, mode, Is), x.device)
    sh = _SharedExpert(_bits(gate_up).value, _bits(down).value, _bits(gate).value, Is)
    _check("moe_forward_shared", lib().moe_forward_shared(
        _bits(x), _bits(router_w), pack.handle, ctypes.byref(sh), T, k, mode, _bits(out),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_quantize_act_nvfp4(x, input_scale: float, codes=None, scales=None, stream=None):
    """NVFP4 quantiser Q of BF16 rows: returns (codes [rows, cols/2] u8, scales [rows, cols/16])."""
    import torch
    rows, cols = x.shape
    if codes is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
    _check("moe_quantize_act_nvfp4", lib().moe_quantize_act_nvfp4(
        _bits(x), rows, cols, float(input_scale), _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def moe_read_device_status(ws, stream=None) -> int:
    """Read and clear a workspace's device status word; ws = None reads the one of
    moe_route_topk_noalloc's fixed array on the current device."""
    st = ctypes.c_int()
    wp = ctypes.c_void_p(None) if ws is None else _ptr(ws)
    _check("moe_read_device_status", lib().moe_read_device_status(wp, _stream(stream),
                                                                  ctypes.byref(st)))
    return st.value


def moe_last_launch_count() -> int:
    return lib().moe_last_launch_count()


def moe_profile_next_forward(events) -> None:
    """Record torch.cuda.Event objects around the kernel launches of the next moe_forward /
    moe_forward_shared call (see the header): events[2i] before and events[2i+1] after the i-th
    launch."""
    arr = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
    _check("moe_profile_next_forward", lib().moe_profile_next_forward(arr, len(events)))


def moe_test_inject_faults(skip_logits_cta: int = -1, wait_limit_seconds: float = 0.0,
                           fail_pack_allocations: int = 0) -> None:
    """Test-only fault injection (see the header); no arguments switch it off."""
    _check("moe_test_inject_faults", lib().moe_test_inject_faults(
        int(skip_logits_cta), float(wait_limit_seconds), int(fail_pack_allocations)))


def moe_profile_kernel_name(i: int):
    """Kernel name of the i-th launch of the last profiled call, or None."""
    n = lib().moe_profile_kernel_name(int(i))
    return None if n is None else n.decode()


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()
