"""Shared helpers of the GPU parity tests: building a layer for both sides, and comparing the
CUDA path with the oracle under the rules the tests state.

Comparison rules:
* top-k indices: bit-exact, except for tokens whose oracle logits have a near tie within the
  FP32 accumulation bound of the GPU router (gamma_n * sum|x*w|); there any selection that is
  a valid top-k under that bound passes, and the token's output is not compared when the
  selected set differs;
* permutation, counts, offsets: bit-exact (they are unique given the selection);
* W4A4 activation codes and scales: bit-exact;
* W4A4 h codes: bit-exact, except elements/blocks the oracle flags as lying within the FP32
  error window of a rounding boundary; each accepted flip widens that token's output bound by
  the oracle's |dh| * ||Wd[:, i]|| for it (triangle inequality);
* W4A8 x codes: bit-exact; W4A8 h codes: bit-exact except elements the oracle flags, each
  accepted difference widening the token's bound by the oracle's largest move of that element;
* outputs: per token ||y - y_ref||_2 <= tol * ||y_ref||_2 (+ the flip allowance), tol = 2e-3
  (W4A16) and 5e-3 (W4A4, W4A8: activations quantised).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import nvfp4_mixture_experts_bf16_gb300 as moe

TOL = {0: 2e-3, 1: 5e-3, 2: 5e-3}
U = 2.0 ** -24
# Summation-depth bounds n of the FP32 router accumulation (error <= gamma(n) * sum|x*w|).
# Narrow calls: per warp one tensor-core chain of 16-product MMA steps over H/8 (16 steps at
# H = 4096, two interleaved chains), then 8 warp partials: n <= 16*16 + 1 + 8 < 300. The
# route-only kernel (FMA tree) is far below that. Wide calls: tcgen05 over 64 K-steps.
GAMMA_NARROW = 300
GAMMA_WIDE = 300


def gamma(n):
    return n * U / (1 - n * U)


def dev_bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(torch.bfloat16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def small_layer(T, H, E, k, I, zipf=False, seed=0, layer=0):
    x = synth.activations(seed, layer, T, H, zipf)
    wr = synth.router_weight(seed, layer, E, H, zipf)
    ex = oracle.ExpertSet(E, H, I)
    xs = synth.activation_input_scale(H)
    ds = synth.down_input_scales(seed, layer, E)
    for e in range(E):
        g = oracle.quantize_weight_bf16(synth.expert_weight(seed, layer, e, "gate", H, I))
        u = oracle.quantize_weight_bf16(synth.expert_weight(seed, layer, e, "up", H, I))
        d = oracle.quantize_weight_bf16(synth.expert_weight(seed, layer, e, "down", H, I))
        ex.set(e, g[:2], u[:2], d[:2], (g[2], u[2], d[2]), (xs, xs, float(ds[e])))
    return x, wr, ex


def pack_from_experts(ex: oracle.ExpertSet) -> moe.Pack:
    mats = []
    for which, lst in ((0, ex.gate), (1, ex.up), (2, ex.down)):
        mats.append([(lst[e][0], lst[e][1], float(ex.mult[e, which]), float(ex.in_scale[e, which]))
                     for e in range(ex.E)])
    return moe.moe_pack_nvfp4(mats[0], mats[1], mats[2], ex.H, ex.I)


class FullLayer:
    """A full-size layer drawn on the device (torch generator) and quantised by the product
    quantiser; the oracle side re-quantises the experts it needs from the same BF16 draws with
    its own quantiser (and the test checks that both quantisers agree bit for bit)."""

    def __init__(self, seed, layer, T, zipf, H=4096, E=512, I=384):
        self.H, self.E, self.I, self.T = H, E, I, T
        self.x = synth.activations(seed, layer, T, H, zipf)
        self.wr = synth.router_weight(seed, layer, E, H, zipf)
        self.xs = synth.activation_input_scale(H)
        self.ds = synth.down_input_scales(seed, layer, E)
        self.W = {w: synth.torch_expert_weights(seed, layer, w, E, H, I, "cuda")
                  for w in ("gate", "up", "down")}
        self.q = {}
        for w, W in self.W.items():
            amax = W.float().abs().amax(dim=(1, 2)).cpu().numpy().astype(np.float32)
            # IEEE float32 division (torch divides a tensor by a scalar via a reciprocal)
            Sh = amax / np.float32(2688.0)
            rows, cols = W.shape[1], W.shape[2]
            codes = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device="cuda")
            scales = torch.empty((E, rows, cols // 16), dtype=torch.uint8, device="cuda")
            for e in range(E):
                moe.moe_quantize_act_nvfp4(W[e], float(Sh[e]), codes[e], scales[e])
            self.q[w] = (codes, scales, Sh)
        torch.cuda.synchronize()
        mats = []
        for wi, w in enumerate(("gate", "up", "down")):
            codes, scales, Sh = self.q[w]
            ins = [self.xs] * E if w != "down" else [float(v) for v in self.ds]
            mats.append([(codes[e], scales[e], float(Sh[e]), ins[e]) for e in range(E)])
        self.pack = moe.moe_pack_nvfp4(mats[0], mats[1], mats[2], H, I)

    def oracle_experts(self, experts, nthreads: int = 8) -> oracle.ExpertSet:
        """ExpertSet with the given experts, quantised by the oracle from the same BF16 draws;
        asserts bit equality with the product quantiser's codes."""
        ex = oracle.ExpertSet(self.E, self.H, self.I)
        ex.in_scale[:, 0] = self.xs       # every expert carries the layer's input scales, also
        ex.in_scale[:, 1] = self.xs       # the ones that are not supplied
        ex.in_scale[:, 2] = self.ds
        for e in sorted(set(int(v) for v in experts)):
            got = {}
            for w in ("gate", "up", "down"):
                wb = host_u16(self.W[w][e])
                c, s, S = oracle.quantize_weight_bf16(wb, nthreads=nthreads)
                gc, gs, gS = self.q[w]
                assert np.float32(S) == np.float32(gS[e]), (w, e)
                assert np.array_equal(c, gc[e].cpu().numpy()), ("codes", w, e)
                assert np.array_equal(s, gs[e].cpu().numpy()), ("scales", w, e)
                got[w] = (c, s, S)
            ex.set(e, got["gate"][:2], got["up"][:2], got["down"][:2],
                   (got["gate"][2], got["up"][2], got["down"][2]),
                   (self.xs, self.xs, float(self.ds[e])))
        return ex

    def close(self):
        self.pack.close()
        self.W = None
        self.q = None


def check_topk(gpu_idx, gpu_w, ref, n_gamma):
    """Returns the tokens whose selected set differs from the oracle's (each validated)."""
    T, k = gpu_idx.shape
    E = ref["logits"].shape[1]
    g = gamma(n_gamma)
    differ = []
    for t in range(T):
        L = ref["logits"][t]
        B = g * ref["abssum"][t]
        sel = gpu_idx[t].astype(np.int64)
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < E, (t, sel)
        if not np.array_equal(sel, ref["idx"][t]):
            for a in range(k - 1):
                assert L[sel[a]] + B[sel[a]] >= L[sel[a + 1]] - B[sel[a + 1]], ("order", t)
            uns = np.setdiff1d(np.arange(E), sel)
            if len(uns):
                assert (L[sel] + B[sel]).min() >= (L[uns] - B[uns]).max(), ("set", t)
            if set(sel.tolist()) != set(ref["idx"][t].tolist()):
                differ.append(t)
        # the weight of each selected expert: softmax of the oracle logits, within the logit
        # error bound (|d log w| <= 2 max|dL|) plus FP32 rounding of exp and the sum
        Lsel = L[sel]
        wref = np.exp(Lsel - Lsel.max())
        wref /= wref.sum()
        rel = np.abs(gpu_w[t] / wref - 1)
        assert rel.max() <= 4 * B.max() + 1e-5, (t, rel.max(), B.max())
    return differ


def stable_perm(idx, E):
    """The unique expert-major, token-stable permutation of a selection (for validity checks
    when the selection differs from the oracle's)."""
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    pairs = sorted((int(idx[t, j]), t) for t in range(T) for j in range(k))
    return counts, offsets, np.array([t for _, t in pairs], np.int32)


def slot_map(perm, offsets):
    """(token, expert) -> slot."""
    m = {}
    E = len(offsets) - 1
    for e in range(E):
        for s in range(offsets[e], offsets[e + 1]):
            m[(int(perm[s]), e)] = s
    return m


def ws_array(ws: torch.Tensor, off: int, nbytes: int, dtype) -> np.ndarray:
    return ws[off:off + nbytes].cpu().numpy().view(dtype)


def h_flip_allowance(gq, gsf, ref, ref_slot, I):
    """Validate the GPU's W4A4 h codes against the oracle's and return the output-error
    allowance (absolute L2) of the accepted flips for that slot."""
    rq, rsf = ref["hq_codes"][ref_slot], ref["hq_scales"][ref_slot]
    allow = 0.0
    flips = 0
    for b in range(I // 16):
        if gsf[b] != rsf[b]:
            assert ref["h_amb_block"][ref_slot, b] > 0, ("unflagged block-scale flip", ref_slot, b)
            allow += ref["h_amb_block"][ref_slot, b]
            flips += 1
            continue
        for i in range(16):
            col = b * 16 + i
            cg = (gq[col // 2] >> (4 * (col % 2))) & 0xF
            cr = (rq[col // 2] >> (4 * (col % 2))) & 0xF
            if cg != cr:
                if (cg & 7) == 0 and (cr & 7) == 0:
                    continue  # +0 / -0
                assert ref["h_amb_elem"][ref_slot, col] > 0, ("unflagged code flip", ref_slot, col)
                allow += ref["h_amb_elem"][ref_slot, col]
                flips += 1
    return allow, flips


def h8_flip_allowance(gq8, ref, ref_slot):
    """Validate the GPU's W4A8 h codes (E4M3 bytes) against the oracle's and return the output
    allowance (absolute L2) of the accepted differences for that slot."""
    rq = ref["hq_codes"][ref_slot]
    allow, flips = 0.0, 0
    for i in np.flatnonzero(gq8 != rq):
        if (gq8[i] & 0x7F) == 0 and (rq[i] & 0x7F) == 0:
            continue  # +0 / -0
        assert ref["h_amb_elem"][ref_slot, i] > 0, ("unflagged E4M3 h difference", ref_slot, i)
        allow += ref["h_amb_elem"][ref_slot, i]
        flips += 1
    return allow, flips


def compare_outputs(out_gpu_u16, ref, mode, tokens, allowance=None):
    """Per-token relative L2 error against the oracle output; returns the max relative error."""
    y = synth.bf16_to_f32(out_gpu_u16).astype(np.float64)
    yr = synth.bf16_to_f32(ref["out_bf16"]).astype(np.float64)
    worst = 0.0
    for t in tokens:
        err = np.linalg.norm(y[t] - yr[t])
        nrm = np.linalg.norm(yr[t])
        extra = 0.0 if allowance is None else allowance.get(t, 0.0)
        assert err <= TOL[mode] * nrm + extra * (1 + 2 ** -7) + 1e-30, \
            (t, err / max(nrm, 1e-300), extra / max(nrm, 1e-300))
        if extra == 0.0:
            worst = max(worst, err / max(nrm, 1e-300))
    return worst
