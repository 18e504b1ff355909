"""CPU oracle for the NVFP4 routed-expert MoE feed-forward step.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The GPU product path
(``nvfp4_mixture_experts_bf16_gb300``) never imports it, and this package never imports the
product.

The arithmetic lives in ``moe_oracle.cpp`` (plain C++, FP64 accumulation, E2M1/E4M3 decoded by
table); this module only compiles it with g++ and marshals numpy arrays through ctypes.

Sources followed (see the C++ header comment for the readings taken where the pages are
silent): the model card "Qwen3.8-Flash-Next NVIDIA NVFP4 for Infernix (bit-exact)", section
"What is bit-exact and what is quantized", and the Infernix README, section "Activation
precision".

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` (exhaustive format
decode against the closed-form definition, brute-force nearest rounding, numpy float32
arithmetic, top-k invariants and closed forms, one-hot / identical-expert / SiLU(0) special
cases and numpy float64 matmuls; the shared expert by equality with a routed expert of the same
weights, scipy's logistic function and closed-form combines). The match of ``quantize_nvfp4`` to NVIDIA's own checkpoint
quantiser is parity unpinned: no checkpoint is available.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

W4A16 = 0
W4A4 = 1
W4A8 = 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmoe_oracle.so`` with g++ (-O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Inputs(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int), ("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
        ("I", ctypes.c_int), ("mode", ctypes.c_int), ("y_keep_fp64", ctypes.c_int),
        ("nthreads", ctypes.c_int), ("amb_eps", ctypes.c_double),
        ("x", ctypes.c_void_p), ("router", ctypes.c_void_p),
        ("gate_codes", ctypes.c_void_p), ("gate_scales", ctypes.c_void_p),
        ("up_codes", ctypes.c_void_p), ("up_scales", ctypes.c_void_p),
        ("down_codes", ctypes.c_void_p), ("down_scales", ctypes.c_void_p),
        ("mult", ctypes.c_void_p), ("in_scale", ctypes.c_void_p),
    ]


_OUT_FIELDS = ["out_bf16", "out64", "logits", "abssum", "idx", "w", "counts", "offsets", "perm",
               "slot_of", "g", "u", "h", "h_bf16", "hq_codes", "hq_scales", "h_amb_elem",
               "h_amb_block", "y", "xq_codes", "xq_scales"]


class _Outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _OUT_FIELDS]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_e2m1_value.argtypes = [ctypes.c_int]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_value.argtypes = [ctypes.c_int]
            L.oracle_e2m1_encode.restype = ctypes.c_int
            L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_int
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_f32_mul.restype = ctypes.c_float
            L.oracle_f32_mul.argtypes = [ctypes.c_float, ctypes.c_float]
            L.oracle_f32_div.restype = ctypes.c_float
            L.oracle_f32_div.argtypes = [ctypes.c_float, ctypes.c_float]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_quantize_nvfp4.restype = None
            L.oracle_quantize_nvfp4.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int]
            L.oracle_quantize_block_steps.restype = None
            L.oracle_quantize_block_steps.argtypes = [ctypes.c_void_p, ctypes.c_float] + \
                [ctypes.c_void_p] * 6
            L.oracle_quantize_weight_bf16.restype = ctypes.c_float
            L.oracle_quantize_weight_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                      ctypes.c_int64, ctypes.c_void_p,
                                                      ctypes.c_void_p, ctypes.c_int]
            L.oracle_dequantize_nvfp4.restype = None
            L.oracle_dequantize_nvfp4.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_double, ctypes.c_void_p]
            L.oracle_route.restype = None
            L.oracle_route.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 4 + \
                [ctypes.c_void_p] * 8 + [ctypes.c_int]
            L.oracle_moe_forward.restype = ctypes.c_int
            L.oracle_moe_forward.argtypes = [ctypes.POINTER(_Inputs), ctypes.POINTER(_Outputs)]
            L.oracle_shared_expert.restype = None
            L.oracle_shared_expert.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 3 + \
                [ctypes.c_void_p] * 8 + [ctypes.c_int]
            L.oracle_moe_forward_shared.restype = ctypes.c_int
            L.oracle_moe_forward_shared.argtypes = [ctypes.POINTER(_Inputs), ctypes.c_int] + \
                [ctypes.c_void_p] * 3 + [ctypes.POINTER(_Outputs)] + [ctypes.c_void_p] * 5
            L.oracle_quantize_a8.restype = None
            L.oracle_quantize_a8.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                             ctypes.c_void_p]
            L.oracle_h8_ambiguity.restype = None
            L.oracle_h8_ambiguity.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.c_double,
                                              ctypes.c_void_p, ctypes.c_void_p]
            L.oracle_h_ambiguity.restype = None
            L.oracle_h_ambiguity.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.c_double,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ format primitives
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(int(byte))


def e2m1_encode(v: float) -> int:
    return lib().oracle_e2m1_encode(float(v))


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(float(v))


def f32_mul(a: float, b: float) -> float:
    return lib().oracle_f32_mul(a, b)


def f32_div(a: float, b: float) -> float:
    return lib().oracle_f32_div(a, b)


def double_to_bf16(v: float) -> int:
    return int(lib().oracle_double_to_bf16(float(v)))


# ------------------------------------------------------------------ quantiser
def quantize_nvfp4(v: np.ndarray, S: float, nthreads: int = 1):
    """Q over the rows of a float32 matrix [rows, cols]; returns (codes [rows, cols/2] uint8,
    scales [rows, cols/16] uint8 E4M3)."""
    v = _c(v, np.float32)
    rows, cols = v.shape
    assert cols % 16 == 0
    codes = np.empty((rows, cols // 2), np.uint8)
    scales = np.empty((rows, cols // 16), np.uint8)
    lib().oracle_quantize_nvfp4(_ptr(v), rows, cols, float(S), _ptr(codes), _ptr(scales),
                                int(nthreads))
    return codes, scales


def quantize_a8(v: np.ndarray, S: float) -> np.ndarray:
    """The W4A8 activation quantiser: E4M3 bytes of float32 values with per-matrix scale S
    (S8 = fl32(6 S), q = E4M3_RNE_satfinite(fl32(v * fl32(1 / S8))), sign kept)."""
    v = _c(v, np.float32)
    codes = np.empty(v.shape, np.uint8)
    lib().oracle_quantize_a8(_ptr(v), v.size, float(S), _ptr(codes))
    return codes


def h8_ambiguity(v16: np.ndarray, S: float, eps: float, colnorm16: np.ndarray) -> np.ndarray:
    """The W4A8 h quantiser's ambiguity for one 16-element block: elem [16] allowances."""
    v = _c(v16, np.float32).reshape(16)
    cn = _c(colnorm16, np.float64).reshape(16)
    elem = np.zeros(16, np.float64)
    lib().oracle_h8_ambiguity(_ptr(v), float(S), float(eps), _ptr(cn), _ptr(elem))
    return elem


def h_ambiguity(v16: np.ndarray, S: float, eps: float, colnorm16: np.ndarray):
    """The W4A4 h quantiser's ambiguity for one 16-element block of FP32 h values with down
    input scale S (see h_ambiguity in moe_oracle.cpp): (elem [16], block) output allowances."""
    v = _c(v16, np.float32).reshape(16)
    cn = _c(colnorm16, np.float64).reshape(16)
    elem = np.zeros(16, np.float64)
    block = np.zeros(1, np.float64)
    lib().oracle_h_ambiguity(_ptr(v), float(S), float(eps), _ptr(cn), _ptr(elem), _ptr(block))
    return elem, float(block[0])


def quantize_block_steps(v16: np.ndarray, S: float) -> dict:
    v16 = _c(v16, np.float32)
    assert v16.shape == (16,)
    inv6S = ctypes.c_float()
    t = ctypes.c_float()
    sf = ctypes.c_int()
    r = ctypes.c_float()
    scaled = np.empty(16, np.float32)
    codes = np.empty(16, np.uint8)
    lib().oracle_quantize_block_steps(_ptr(v16), float(S), ctypes.byref(inv6S), ctypes.byref(t),
                                      ctypes.byref(sf), ctypes.byref(r), _ptr(scaled),
                                      _ptr(codes))
    return dict(inv6S=inv6S.value, t=t.value, sf=sf.value, r=r.value, scaled=scaled,
                codes=codes)


def quantize_weight_bf16(w_bf16: np.ndarray, nthreads: int = 1):
    """Quantise a BF16 weight matrix (uint16 bit patterns [rows, cols]) the way the synthetic
    checkpoints are made; returns (codes, scales, multiplier)."""
    w = _c(w_bf16, np.uint16)
    rows, cols = w.shape
    codes = np.empty((rows, cols // 2), np.uint8)
    scales = np.empty((rows, cols // 16), np.uint8)
    S = lib().oracle_quantize_weight_bf16(_ptr(w), rows, cols, _ptr(codes), _ptr(scales),
                                          int(nthreads))
    return codes, scales, float(np.float32(S))


def dequantize_nvfp4(codes: np.ndarray, scales: np.ndarray, mult: float) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    out = np.empty((rows, cols), np.float64)
    lib().oracle_dequantize_nvfp4(_ptr(codes), _ptr(scales), rows, cols, float(mult), _ptr(out))
    return out


# ------------------------------------------------------------------ routing
def route(x_bf16: np.ndarray, wr_bf16: np.ndarray, k: int, nthreads: int = 1) -> dict:
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    T, H = x.shape
    E = wr.shape[0]
    logits = np.empty((T, E), np.float64)
    abssum = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    slot_of = np.empty((T, k), np.int32)
    lib().oracle_route(_ptr(x), _ptr(wr), T, H, E, k, _ptr(logits), _ptr(abssum), _ptr(idx),
                       _ptr(w), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(slot_of),
                       int(nthreads))
    return dict(logits=logits, abssum=abssum, idx=idx, w=w, counts=counts, offsets=offsets,
                perm=perm, slot_of=slot_of)


# ------------------------------------------------------------------ forward
class ExpertSet:
    """Per-expert NVFP4 matrices in checkpoint layout; any expert may be None (not supplied)."""

    def __init__(self, E: int, H: int, I: int):
        self.E, self.H, self.I = E, H, I
        self.gate = [None] * E   # (codes [I, H/2], scales [I, H/16])
        self.up = [None] * E
        self.down = [None] * E   # (codes [H, I/2], scales [H, I/16])
        self.mult = np.ones((E, 3), np.float32)
        self.in_scale = np.ones((E, 3), np.float32)

    def set(self, e, gate, up, down, mult, in_scale=(1.0, 1.0, 1.0)):
        self.gate[e] = tuple(_c(a, np.uint8) for a in gate)
        self.up[e] = tuple(_c(a, np.uint8) for a in up)
        self.down[e] = tuple(_c(a, np.uint8) for a in down)
        self.mult[e] = mult
        self.in_scale[e] = in_scale


class SharedExpert:
    """The BF16 shared expert of a layer (uint16 bit patterns): ``gate_up`` [2*Is, H] (rows
    0..Is-1 gate, Is..2*Is-1 up), ``down`` [H, Is] and the gate vector ``gate`` [H]."""

    def __init__(self, gate_up: np.ndarray, down: np.ndarray, gate: np.ndarray):
        self.gate_up = _c(gate_up, np.uint16)
        self.down = _c(down, np.uint16)
        self.gate = _c(gate, np.uint16).reshape(-1)
        self.Is = self.gate_up.shape[0] // 2
        H = self.gate.shape[0]
        assert self.gate_up.shape == (2 * self.Is, H) and self.down.shape == (H, self.Is)


def shared_expert(x_bf16: np.ndarray, shared: SharedExpert, nthreads: int = 1) -> dict:
    """The shared expert alone: sigma [T] (the gate), hs_bf16 [T, Is], h64 [T, Is] (h before
    its BF16 rounding), ys [T, H] (the down product rounded to BF16, as FP64 values) and ys64
    [T, H] (the down product before that rounding)."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    Is = shared.Is
    sigma = np.empty(T, np.float64)
    hs = np.empty((T, Is), np.uint16)
    h64 = np.empty((T, Is), np.float64)
    ys = np.empty((T, H), np.float64)
    ys64 = np.empty((T, H), np.float64)
    lib().oracle_shared_expert(_ptr(x), T, H, Is, _ptr(shared.gate_up), _ptr(shared.down),
                               _ptr(shared.gate), _ptr(sigma), _ptr(hs), _ptr(ys), _ptr(ys64),
                               _ptr(h64), int(nthreads))
    return dict(sigma=sigma, hs_bf16=hs, h64=h64, ys=ys, ys64=ys64)


def forward(x_bf16: np.ndarray, wr_bf16: np.ndarray, experts: ExpertSet, k: int, mode: int,
            nthreads: int = 1, y_keep_fp64: bool = False, amb_eps: float = 2.0 ** -14,
            want=("out_bf16", "out64", "idx", "w", "perm", "counts", "offsets", "slot_of",
                  "logits", "abssum"), shared: SharedExpert | None = None) -> dict:
    """Run the oracle forward; ``want`` names the outputs to return (see moe_oracle.cpp). With
    ``shared``, the shared expert's gated output is added before the final rounding (out_bf16
    and out64 include it) and sigma, hs_bf16, hs64 (h before its rounding), ys (the down product
    rounded to BF16) and ys64 (before that rounding)
    are returned too."""
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    T, H = x.shape
    E, I = experts.E, experts.I
    assert wr.shape == (E, H) and experts.H == H
    S = T * k

    def ptr_array(lst, j):
        arr = (ctypes.c_void_p * E)()
        for e in range(E):
            arr[e] = None if lst[e] is None else lst[e][j].ctypes.data
        return arr

    keep = [ptr_array(experts.gate, 0), ptr_array(experts.gate, 1), ptr_array(experts.up, 0),
            ptr_array(experts.up, 1), ptr_array(experts.down, 0), ptr_array(experts.down, 1)]
    mult = _c(experts.mult, np.float32)
    ins = _c(experts.in_scale, np.float32)
    inp = _Inputs(T, H, E, k, I, int(mode), int(bool(y_keep_fp64)), int(nthreads),
                  float(amb_eps), _ptr(x), _ptr(wr),
                  *[ctypes.cast(a, ctypes.c_void_p) for a in keep], _ptr(mult), _ptr(ins))
    shapes = dict(out_bf16=((T, H), np.uint16), out64=((T, H), np.float64),
                  logits=((T, E), np.float64), abssum=((T, E), np.float64),
                  idx=((T, k), np.int32), w=((T, k), np.float64), counts=((E,), np.int32),
                  offsets=((E + 1,), np.int32), perm=((S,), np.int32),
                  slot_of=((T, k), np.int32), g=((S, I), np.float64), u=((S, I), np.float64),
                  h=((S, I), np.float64), h_bf16=((S, I), np.uint16),
                  hq_codes=((S, I if mode == 2 else I // 2), np.uint8),
                  hq_scales=((S, I // 16), np.uint8),
                  h_amb_elem=((S, I), np.float64), h_amb_block=((S, I // 16), np.float64),
                  y=((S, H), np.float64),
                  xq_codes=((T, H if mode == 2 else H // 2), np.uint8),
                  xq_scales=((T, H // 16), np.uint8))
    res = {}
    for name in set(want) | {"out_bf16"}:
        shp, dt = shapes[name]
        res[name] = np.zeros(shp, dt)
    outs = _Outputs(*[_ptr(res.get(n)) for n in _OUT_FIELDS])
    if shared is None:
        rc = lib().oracle_moe_forward(ctypes.byref(inp), ctypes.byref(outs))
    else:
        assert shared.gate.shape[0] == H
        res["sigma"] = np.empty(T, np.float64)
        res["hs_bf16"] = np.empty((T, shared.Is), np.uint16)
        res["hs64"] = np.empty((T, shared.Is), np.float64)
        res["ys"] = np.empty((T, H), np.float64)
        res["ys64"] = np.empty((T, H), np.float64)
        rc = lib().oracle_moe_forward_shared(
            ctypes.byref(inp), shared.Is, _ptr(shared.gate_up), _ptr(shared.down),
            _ptr(shared.gate), ctypes.byref(outs), _ptr(res["sigma"]), _ptr(res["hs_bf16"]),
            _ptr(res["ys"]), _ptr(res["ys64"]), _ptr(res["hs64"]))
    if rc != 0:
        raise ValueError(f"oracle forward failed with code {rc}")
    return res
