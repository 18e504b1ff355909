"""Seeded synthetic inputs for the NVFP4 routed-expert MoE step.

This module serves both the GPU path and the oracle. It holds random draws and data shaping
only: no NVFP4 quantisation, routing, SiLU or expert arithmetic (those belong to the oracle and
to the CUDA library). Weights come out as BF16 bit patterns *before* quantisation; each side
quantises them with its own quantiser.

Every tensor is drawn from its own counter-based stream: Philox-4x32-10 (Salmon, Moraes, Dror,
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11), keyed by splitmix64 of
(seed, layer, tensor id, expert). So any one expert can be regenerated alone, in any order and on
any thread, which is what lets a test rebuild only the experts a sampled token selects.

Workloads (sizes from the routed-expert topology on the model card "Qwen3.8-Flash-Next NVIDIA
NVFP4 for Infernix (bit-exact)": 512 routed experts, top-10, 48 layers; hidden 4096 and expert
intermediate 384 are the plainest reading consistent with its ~2.6 MiB per expert):

* ``tiny``          T=4,    H=256,  E=16,  k=2,  I=64,  W4A16, 1 layer
* ``decode1``       T=1,    H=4096, E=512, k=10, I=384, W4A16, 48 layers, near-uniform routing
* ``verify8``       T=8,    same shapes, W4A16, Zipf(1.1) expert popularity
* ``verify8_w4a4``  T=8,    same, W4A4
* ``prefill8192``   T=8192, same, W4A4 (and W4A16 for comparison), Zipf(1.1)

Shared expert (optional): BF16 gate/up [2*Is, H], down [H, Is] and gate vector [H], all
~ N(0, 0.02); the workloads take Is = I.

Value recipe: activations BF16 ~ N(0, 1); router BF16 ~ N(0, 0.02); expert weights
~ N(0, 0.02) rounded to BF16 and then quantised (multiplier = global amax / (6*448), block scale
= E4M3 of block amax / (6 * multiplier)). Zipf workloads add a per-layer expert bias through a
shared direction u (unit vector): x_t = z_t + c*u and Wr[e] = G_e + (b_e / c) * u with c = 8 and
b_e = -LAMBDA * 1.1 * ln(rank_e), rank_e a seeded permutation of 1..E. The W4A4 activation input
scale is amax of a separate 256-token N(0,1) calibration batch (seed 1) over 6*448; the down
projection's input scale per expert is A_e / (6*448) with A_e drawn uniformly in [DOWN_AMAX_LO,
DOWN_AMAX_HI] (a synthetic checkpoint constant; the range brackets the amax of h that a
256-token calibration pass through an expert of this distribution produces).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

MASK64 = (1 << 64) - 1

# Zipf bias strength: fixed once so that the 8192-token workload's busiest expert receives
# about 2000 of the 81,920 routed slots at seed 0.
LAMBDA = 0.30
ZIPF_S = 1.1
ZIPF_C = 8.0
DOWN_AMAX_LO = 12.0
DOWN_AMAX_HI = 19.0
WEIGHT_STD = 0.02
ROUTER_STD = 0.02

# tensor ids for the stream keys
_T_X, _T_ROUTER, _T_GATE, _T_UP, _T_DOWN, _T_CAL, _T_U, _T_PERM, _T_DSCALE = range(1, 10)
_T_SH_GU, _T_SH_DOWN, _T_SH_GATE = range(10, 13)
_WHICH = {"gate": _T_GATE, "up": _T_UP, "down": _T_DOWN}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    mode: int          # 0 = W4A16, 1 = W4A4
    layers: int
    zipf: bool


WORKLOADS = {
    "tiny": Workload("tiny", 4, 256, 16, 2, 64, 0, 1, False),
    "decode1": Workload("decode1", 1, 4096, 512, 10, 384, 0, 48, False),
    "verify8": Workload("verify8", 8, 4096, 512, 10, 384, 0, 48, True),
    "verify8_w4a4": Workload("verify8_w4a4", 8, 4096, 512, 10, 384, 1, 48, True),
    "verify8_w4a8": Workload("verify8_w4a8", 8, 4096, 512, 10, 384, 2, 48, True),
    "prefill8192": Workload("prefill8192", 8192, 4096, 512, 10, 384, 1, 1, True),
}


def splitmix64(x: int) -> int:
    """splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA'14)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, *parts: int) -> int:
    """A 128-bit Philox key from (seed, parts...)."""
    h = splitmix64(seed & MASK64)
    for p in parts:
        h = splitmix64(h ^ (p & MASK64))
    lo = splitmix64(h ^ 0x1234567)
    return (h << 64) | lo


def stream(seed: int, *parts: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=stream_key(seed, *parts)))


def torch_seed(seed: int, *parts: int) -> int:
    """A 63-bit seed for a torch generator derived the same way (device-side generation)."""
    return stream_key(seed, *parts) & ((1 << 63) - 1)


# ------------------------------------------------------------------ BF16 bit patterns
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ draws
def _unit_vector(seed: int, layer: int, H: int) -> np.ndarray:
    n = stream(seed, layer, _T_U).standard_normal(H)
    return n / np.linalg.norm(n)


def zipf_bias(seed: int, layer: int, E: int) -> np.ndarray:
    """b_e = -LAMBDA * s * ln(rank_e), rank_e a seeded permutation of 1..E (float64 [E])."""
    rank = stream(seed, layer, _T_PERM).permutation(E) + 1
    return -LAMBDA * ZIPF_S * np.log(rank.astype(np.float64))


def activations(seed: int, layer: int, T: int, H: int, zipf: bool = False) -> np.ndarray:
    """BF16 [T, H]: N(0,1), plus c*u along the layer's bias direction for Zipf workloads."""
    z = stream(seed, layer, _T_X, T).standard_normal((T, H))
    if zipf:
        z = z + ZIPF_C * _unit_vector(seed, layer, H)[None, :]
    return bf16_bits(z.astype(np.float32))


def router_weight(seed: int, layer: int, E: int, H: int, zipf: bool = False) -> np.ndarray:
    """BF16 [E, H]: N(0, 0.02), plus (b_e / c) * u for Zipf workloads."""
    g = stream(seed, layer, _T_ROUTER).standard_normal((E, H)) * ROUTER_STD
    if zipf:
        b = zipf_bias(seed, layer, E)
        g = g + (b / ZIPF_C)[:, None] * _unit_vector(seed, layer, H)[None, :]
    return bf16_bits(g.astype(np.float32))


def expert_weight(seed: int, layer: int, e: int, which: str, H: int, I: int) -> np.ndarray:
    """BF16 pre-quantisation weights of one expert matrix: gate/up [I, H], down [H, I]."""
    shape = (H, I) if which == "down" else (I, H)
    w = stream(seed, layer, _WHICH[which], e).standard_normal(shape, dtype=np.float32)
    return bf16_bits(w * np.float32(WEIGHT_STD))


def calibration_batch(H: int, seed: int = 1, T: int = 256) -> np.ndarray:
    """BF16 [T, H] ~ N(0, 1): the separate batch the activation input scale is taken from."""
    return bf16_bits(stream(seed, 0, _T_CAL).standard_normal((T, H)).astype(np.float32))


def activation_input_scale(H: int, seed: int = 1) -> float:
    """fl32(amax(calibration batch) / 2688), 2688 = 6 * 448."""
    amax = np.float32(np.abs(bf16_to_f32(calibration_batch(H, seed))).max())
    return float(np.float32(amax) / np.float32(2688.0))


def down_input_scales(seed: int, layer: int, E: int) -> np.ndarray:
    """float32 [E]: A_e / 2688 with A_e ~ U[DOWN_AMAX_LO, DOWN_AMAX_HI]."""
    a = stream(seed, layer, _T_DSCALE).uniform(DOWN_AMAX_LO, DOWN_AMAX_HI, E).astype(np.float32)
    return (a / np.float32(2688.0)).astype(np.float32)


def shared_expert_weights(seed: int, layer: int, H: int, Is: int):
    """The BF16 shared expert of a layer: gate_up [2*Is, H] (gate rows, then up rows), down
    [H, Is] and the gate vector [H], each ~ N(0, 0.02) rounded to BF16."""
    gu = stream(seed, layer, _T_SH_GU).standard_normal((2 * Is, H), dtype=np.float32)
    dn = stream(seed, layer, _T_SH_DOWN).standard_normal((H, Is), dtype=np.float32)
    gv = stream(seed, layer, _T_SH_GATE).standard_normal(H, dtype=np.float32)
    sd = np.float32(WEIGHT_STD)
    return bf16_bits(gu * sd), bf16_bits(dn * sd), bf16_bits(gv * sd)


# ------------------------------------------------------------------ device-side draws
def torch_expert_weights(seed: int, layer: int, which: str, E: int, H: int, I: int, device,
                         experts=None):
    """BF16 torch tensor [E, rows, cols] of pre-quantisation weights drawn on ``device`` with a
    seeded torch generator (a different stream from the numpy one: used by the full-size
    workloads, where both the GPU path and the oracle read the same drawn tensor)."""
    import torch
    rows, cols = (H, I) if which == "down" else (I, H)
    gen = torch.Generator(device=device)
    gen.manual_seed(torch_seed(seed, layer, _WHICH[which]))
    n = E if experts is None else experts
    w = torch.randn((n, rows, cols), generator=gen, device=device, dtype=torch.float32)
    return (w * WEIGHT_STD).to(torch.bfloat16)


def torch_shared_expert_weights(seed: int, layer: int, H: int, Is: int, device):
    """The shared expert's BF16 weights (gate_up [2*Is, H], down [H, Is], gate [H]) drawn on
    ``device`` with seeded torch generators (the full-size workloads' stream)."""
    import torch
    out = []
    for tid, shape in ((_T_SH_GU, (2 * Is, H)), (_T_SH_DOWN, (H, Is)), (_T_SH_GATE, (H,))):
        gen = torch.Generator(device=device)
        gen.manual_seed(torch_seed(seed, layer, tid))
        w = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        out.append((w * WEIGHT_STD).to(torch.bfloat16))
    return tuple(out)


def describe() -> str:
    return ("seeded synthetic: x~N(0,1) BF16, router~N(0,0.02) BF16, experts~N(0,0.02)->BF16"
            "->NVFP4; Zipf(1.1) bias via shared direction for verify/prefill workloads")


__all__ = [n for n in dir() if not n.startswith("_")]
_ = math
