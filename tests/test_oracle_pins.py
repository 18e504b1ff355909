"""Pins for the CPU oracle, against what the format definitions and the mathematics fix.

Each test ties one oracle function to something other than itself: the closed-form definition
of a format, a printed landmark value (tests/golden), IEEE float32 arithmetic as numpy performs
it, a library routine (numpy matmul, scipy softmax), an invariant, or a closed-form special
case. A plausible slip in the oracle (a dropped term, a wrong sign, a transposed operand, a
wrong tie rule) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_formats.txt")


# ------------------------------------------------------------------ formats
def _e2m1_closed(code):
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return s * mag


def _e4m3_closed(byte):
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 7
    if e == 15 and m == 7:
        return math.nan
    mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return s * mag


def test_e2m1_exhaustive_decode_matches_closed_form():
    for code in range(16):
        assert oracle.e2m1_value(code) == _e2m1_closed(code)


def test_e4m3_exhaustive_decode_matches_closed_form():
    for b in range(256):
        v, ref = oracle.e4m3_value(b), _e4m3_closed(b)
        if math.isnan(ref):
            assert math.isnan(v)
        else:
            assert v == ref and math.copysign(1, v) == math.copysign(1, ref)


def test_formats_golden_landmarks():
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        code = int(code, 16)
        got = oracle.e2m1_value(code) if fmt == "e2m1" else oracle.e4m3_value(code)
        if val == "nan":
            assert math.isnan(got)
        else:
            ref = float(val)
            assert got == ref and math.copysign(1, got) == math.copysign(1, ref), (fmt, code)
        n += 1
    assert n == 26


def _nearest_brute(values, v, codes):
    """Nearest representable magnitude by exhaustive search, ties to the even code."""
    best = None
    for c, m in zip(codes, values):
        d = abs(m - abs(v))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return best[1]


def test_e2m1_encode_textbook_ties_and_saturation():
    # ties go to the even code (RNE), values above 6 saturate to 6
    cases = [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
             (5.0, 0x6), (0.2499, 0x0), (0.2501, 0x1), (5.0001, 0x7), (6.0, 0x7), (7.0, 0x7),
             (1e30, 0x7), (-0.75, 0xA), (-1e-9, 0x8), (0.0, 0x0), (-0.0, 0x8)]
    for v, c in cases:
        assert oracle.e2m1_encode(v) == c, v


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(1)
    mags = [abs(_e2m1_closed(c)) for c in range(8)]
    vals = list(rng.uniform(-7, 7, 400).astype(np.float32))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        for d in (-1, 0, 1):
            vals.append(np.nextafter(np.float32(m), np.float32(np.inf if d > 0 else -np.inf))
                        if d else np.float32(m))
    for v in vals:
        v = float(np.float32(v))
        want = _nearest_brute(mags, min(abs(v), 6.0), list(range(8)))
        want |= 8 if math.copysign(1, v) < 0 else 0
        assert oracle.e2m1_encode(v) == want, v


def test_e4m3_encode_brute_force_and_ties():
    mags = [_e4m3_closed(b) for b in range(0x7F)]
    rng = np.random.default_rng(2)
    vals = list(np.exp(rng.uniform(np.log(1e-4), np.log(500), 500)).astype(np.float32))
    for b in range(0x7E):   # every midpoint and its float neighbours
        mid = np.float32((mags[b] + mags[b + 1]) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    for v in vals:
        v = float(v)
        want = 0x7E if v >= 448 else _nearest_brute(mags, v, list(range(0x7F)))
        assert oracle.e4m3_encode(v) == want, v
    assert oracle.e4m3_encode(1.0625) == 0x38   # tie between 1 (0x38) and 1.125 -> even
    assert oracle.e4m3_encode(1.1875) == 0x3A   # tie between 1.125 and 1.25 -> even
    assert oracle.e4m3_encode(2.0 ** -10) == 0  # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(464.0) == 0x7E    # satfinite
    assert oracle.e4m3_encode(1e30) == 0x7E


def test_f32_ops_match_numpy_ieee_float32():
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(3000) * np.exp(rng.uniform(-60, 60, 3000))).astype(np.float32)
    b = (rng.standard_normal(3000) * np.exp(rng.uniform(-60, 60, 3000))).astype(np.float32)
    a[:10] = np.float32(1e-42)   # subnormals
    with np.errstate(all="ignore"):
        pm = a * b
        pd = a / b
    for i in range(len(a)):
        m = oracle.f32_mul(float(a[i]), float(b[i]))
        d = oracle.f32_div(float(a[i]), float(b[i]))
        assert np.float32(m).tobytes() == pm[i].tobytes()
        assert np.float32(d).tobytes() == pd[i].tobytes()


def test_double_to_bf16_against_independent_rounding():
    rng = np.random.default_rng(4)
    f = (rng.standard_normal(5000) * np.exp(rng.uniform(-30, 30, 5000))).astype(np.float32)
    ref = synth.bf16_bits(f)   # integer rounding of the float32 pattern
    got = np.array([oracle.double_to_bf16(float(v)) for v in f], np.uint16)
    assert np.array_equal(ref, got)
    # ties in double precision: exactly halfway between two BF16 values
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80            # tie -> even (1.0)
    assert oracle.double_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82        # tie -> even
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81  # just above the tie


# ------------------------------------------------------------------ quantiser
def test_quantizer_steps_match_numpy_float32():
    rng = np.random.default_rng(5)
    for _ in range(200):
        S = np.float32(np.exp(rng.uniform(-12, 2)))
        v = (rng.standard_normal(16) * np.exp(rng.uniform(-3, 3))).astype(np.float32)
        st = oracle.quantize_block_steps(v, float(S))
        inv6S = np.float32(1) / (np.float32(6) * S)
        assert np.float32(st["inv6S"]) == inv6S
        t = np.float32(np.abs(v).max()) * inv6S
        assert np.float32(st["t"]) == t
        assert st["sf"] == oracle.e4m3_encode(float(t))
        sfv = np.float32(oracle.e4m3_value(st["sf"]))
        if sfv == 0:
            assert np.all(st["codes"] == 0)
            continue
        r = np.float32(1) / (sfv * S)
        assert np.float32(st["r"]) == r
        assert np.array_equal(st["scaled"], v * r)
        for i in range(16):
            assert st["codes"][i] == oracle.e2m1_encode(float(v[i] * r))


def _dec_block(codes, sf, S):
    return np.array([oracle.e2m1_value(c) for c in codes]) * oracle.e4m3_value(sf) * S


def test_quantizer_round_trip_on_representable_blocks():
    rng = np.random.default_rng(6)
    for _ in range(300):
        S = float(np.float32(np.exp(rng.uniform(-12, 0))))
        sf = int(rng.integers(0x08, 0x7E))          # a normal, unsaturated scale
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = 7 | (8 * int(rng.integers(0, 2)))   # the amax -> 6
        v = _dec_block(codes, sf, S).astype(np.float32)
        if not np.all(v.astype(np.float64) == _dec_block(codes, sf, S)):
            continue   # not exactly representable in float32 at this S
        c, s = oracle.quantize_nvfp4(v[None, :], S)
        assert s[0, 0] == sf
        dec_codes = [(c[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
        # zero codes may carry either sign; compare decoded values for them
        assert np.array_equal(_dec_block(dec_codes, sf, S), _dec_block(codes, sf, S))


def test_quantizer_error_and_amax_invariants():
    rng = np.random.default_rng(7)
    rows = (rng.standard_normal((200, 64)) * np.exp(rng.uniform(-2, 2, (200, 1)))).astype(
        np.float32)
    S = float(np.float32(np.abs(rows).max() / 2688.0))
    codes, scales = oracle.quantize_nvfp4(rows, S)
    for r in range(rows.shape[0]):
        for b in range(4):
            v = rows[r, b * 16:(b + 1) * 16].astype(np.float64)
            sf = scales[r, b]
            cs = [(codes[r, b * 8 + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
            dec = _dec_block(cs, sf, S)
            unit = oracle.e4m3_value(sf) * S
            # every element within half a step of the grid it was rounded on (steps 0.5/1/2)
            for i in range(16):
                mag = abs(v[i]) / unit
                step = 0.5 if mag <= 2 else (1.0 if mag <= 4 else 2.0)
                assert abs(dec[i] - v[i]) <= (step / 2) * unit * (1 + 1e-6) + 1e-30
                assert np.sign(dec[i]) in (0, np.sign(v[i]))
            amax_i = int(np.argmax(np.abs(v)))
            if 0x08 <= sf < 0x7E:
                assert cs[amax_i] & 7 == 7     # the block maximum maps to +-6


def test_quantizer_zero_and_saturated_blocks():
    c, s = oracle.quantize_nvfp4(np.zeros((1, 16), np.float32), 0.01)
    assert s[0, 0] == 0 and np.all(c == 0)
    v = np.full((1, 16), 1e6, np.float32)
    v[0, 3] = -1e6
    c, s = oracle.quantize_nvfp4(v, 1e-3)
    assert s[0, 0] == 0x7E
    assert c[0, 0] == 0x77 and c[0, 1] == 0xF7


# ------------------------------------------------------------------ routing
def _tiny_route_inputs(seed, T, E, H):
    x = synth.activations(seed, 0, T, H)
    wr = synth.router_weight(seed, 0, E, H)
    return x, wr


def test_route_topk_brute_force_and_tie_rule():
    T, E, H, k = 5, 9, 64, 3
    x, wr = _tiny_route_inputs(11, T, E, H)
    wr[4] = wr[2]     # experts 2 and 4 have equal logits: 2 must come first
    wr[7] = wr[2]
    r = oracle.route(x, wr, k)
    l64 = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(wr).astype(np.float64).T
    assert np.allclose(r["logits"], l64, rtol=1e-13, atol=1e-13)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-l64[t, e], e))
        assert list(r["idx"][t]) == order[:k]
        sel = set(order[:k])
        assert min(l64[t, e] for e in sel) >= max(l64[t, e] for e in range(E) if e not in sel)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, rtol=1e-14)
    for t in range(T):
        for a in range(k):
            for b in range(k):
                ia, ib = r["idx"][t, a], r["idx"][t, b]
                assert math.isclose(r["w"][t, a] / r["w"][t, b],
                                    math.exp(l64[t, ia] - l64[t, ib]), rel_tol=1e-12)


def test_route_k1_and_k_equals_E():
    T, E, H = 4, 6, 32
    x, wr = _tiny_route_inputs(12, T, E, H)
    r1 = oracle.route(x, wr, 1)
    assert np.all(r1["w"] == 1.0)
    rE = oracle.route(x, wr, E)
    full = softmax(rE["logits"], axis=1)
    for t in range(T):
        np.testing.assert_allclose(rE["w"][t], full[t, rE["idx"][t]], rtol=1e-13)


def test_route_permutation_is_a_stable_counting_sort():
    T, E, H, k = 37, 16, 64, 4
    x, wr = _tiny_route_inputs(13, T, E, H)
    r = oracle.route(x, wr, k)
    assert r["counts"].sum() == T * k
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
    pairs = sorted((int(r["idx"][t, j]), t) for t in range(T) for j in range(k))
    assert list(r["perm"]) == [t for _, t in pairs]
    for t in range(T):
        for j in range(k):
            s = r["slot_of"][t, j]
            e = r["idx"][t, j]
            assert r["perm"][s] == t and r["offsets"][e] <= s < r["offsets"][e + 1]
    assert sorted(r["slot_of"].ravel().tolist()) == list(range(T * k))


# ------------------------------------------------------------------ expert FFN
def _make_experts(seed, E, H, I, down_scales=None):
    ex = oracle.ExpertSet(E, H, I)
    for e in range(E):
        gq = oracle.quantize_weight_bf16(synth.expert_weight(seed, 0, e, "gate", H, I))
        uq = oracle.quantize_weight_bf16(synth.expert_weight(seed, 0, e, "up", H, I))
        dq = oracle.quantize_weight_bf16(synth.expert_weight(seed, 0, e, "down", H, I))
        xs = synth.activation_input_scale(H)
        ds = 14.0 / 2688 if down_scales is None else down_scales[e]
        ex.set(e, gq[:2], uq[:2], dq[:2], (gq[2], uq[2], dq[2]), (xs, xs, ds))
    return ex


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    x = synth.activations(0, 0, wl.T, wl.H)
    wr = synth.router_weight(0, 0, wl.E, wl.H)
    ex = _make_experts(0, wl.E, wl.H, wl.I, synth.down_input_scales(0, 0, wl.E))
    return wl, x, wr, ex


def test_forward_matches_numpy_float64_pipeline(tiny):
    wl, x, wr, ex = tiny
    res = oracle.forward(x, wr, ex, wl.k, oracle.W4A16,
                         want=("out64", "idx", "w", "slot_of", "perm", "g", "u", "h", "y"))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    for s in range(wl.T * wl.k):
        t = res["perm"][s]
        e = int(np.searchsorted(np.cumsum(np.bincount(res["idx"].ravel(), minlength=wl.E)), s,
                                side="right"))
        Wg = oracle.dequantize_nvfp4(*ex.gate[e], ex.mult[e, 0])
        Wu = oracle.dequantize_nvfp4(*ex.up[e], ex.mult[e, 1])
        Wd = oracle.dequantize_nvfp4(*ex.down[e], ex.mult[e, 2])
        g = Wg @ xf[t]
        u = Wu @ xf[t]
        np.testing.assert_allclose(res["g"][s], g, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(res["u"][s], u, rtol=1e-12, atol=1e-12)
        h = g * (1 / (1 + np.exp(-g))) * u
        np.testing.assert_allclose(res["h"][s], h, rtol=1e-12, atol=1e-12)
        hb = synth.bf16_to_f32(np.array([oracle.double_to_bf16(v) for v in h], np.uint16))
        y = Wd @ hb.astype(np.float64)
        yb = synth.bf16_to_f32(np.array([oracle.double_to_bf16(v) for v in y], np.uint16))
        np.testing.assert_allclose(res["y"][s], yb, rtol=0, atol=0)
    for t in range(wl.T):
        acc = sum(res["w"][t, j] * res["y"][res["slot_of"][t, j]] for j in range(wl.k))
        np.testing.assert_allclose(res["out64"][t], acc, rtol=1e-13, atol=1e-13)


def test_forward_one_hot_weights_closed_form():
    E, H, I, k, T = 4, 64, 32, 1, 3
    x = synth.activations(21, 0, T, H)
    wr = synth.router_weight(21, 0, E, H)
    ex = oracle.ExpertSet(E, H, I)
    rng = np.random.default_rng(21)
    sf = 0x38   # scale 1.0
    for e in range(E):
        cols = rng.integers(0, H, I)
        gc = np.zeros((I, H // 2), np.uint8)
        for i in range(I):
            c = cols[i]
            gc[i, c // 2] |= 7 << (4 * (c % 2))      # code +6 at one column per row
        gs = np.full((I, H // 16), sf, np.uint8)
        ex.set(e, (gc, gs), (gc, gs), (np.zeros((H, I // 2), np.uint8),
                                        np.zeros((H, I // 16), np.uint8)), (0.25, 0.5, 1.0))
        ex.cols = getattr(ex, "cols", {})
        ex.cols[e] = cols
    res = oracle.forward(x, wr, ex, k, oracle.W4A16, want=("g", "u", "perm", "idx", "counts"))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    offs = np.concatenate([[0], np.cumsum(res["counts"])])
    for s in range(T * k):
        t = res["perm"][s]
        e = int(np.searchsorted(offs, s, side="right") - 1)
        np.testing.assert_array_equal(res["g"][s], 6 * 0.25 * xf[t, ex.cols[e]])
        np.testing.assert_array_equal(res["u"][s], 6 * 0.5 * xf[t, ex.cols[e]])


def test_forward_identical_experts_give_one_expert(tiny):
    wl, x, wr, ex = tiny
    same = oracle.ExpertSet(wl.E, wl.H, wl.I)
    for e in range(wl.E):
        same.set(e, ex.gate[0], ex.up[0], ex.down[0], ex.mult[0], ex.in_scale[0])
    res = oracle.forward(x, wr, same, wl.k, oracle.W4A16, want=("y", "slot_of"))
    for t in range(wl.T):
        y0 = res["y"][res["slot_of"][t, 0]]
        assert np.array_equal(synth.bf16_to_f32(res["out_bf16"][t]).astype(np.float64), y0)


def test_forward_zero_gate_gives_zero(tiny):
    wl, x, wr, ex = tiny
    z = oracle.ExpertSet(wl.E, wl.H, wl.I)
    zc = (np.zeros((wl.I, wl.H // 2), np.uint8), np.zeros((wl.I, wl.H // 16), np.uint8))
    for e in range(wl.E):
        z.set(e, zc, ex.up[e], ex.down[e], ex.mult[e], ex.in_scale[e])
    res = oracle.forward(x, wr, z, wl.k, oracle.W4A16, want=("h",))
    assert np.all(res["h"] == 0) and np.all(synth.bf16_to_f32(res["out_bf16"]) == 0)


def test_forward_w4a4_equals_w4a16_before_h_on_representable_x(tiny):
    wl, _, wr, ex0 = tiny
    rng = np.random.default_rng(31)
    S = 2.0 ** -9          # a power of two, so code * scale * S is exactly BF16
    ex = oracle.ExpertSet(wl.E, wl.H, wl.I)
    for e in range(wl.E):
        ex.set(e, ex0.gate[e], ex0.up[e], ex0.down[e], ex0.mult[e],
               (S, S, ex0.in_scale[e, 2]))
    codes = rng.integers(0, 16, (wl.T, wl.H))
    codes[:, ::16] = 7
    sfs = rng.integers(0x30, 0x48, (wl.T, wl.H // 16))
    xv = np.array([[oracle.e2m1_value(c) for c in row] for row in codes]) * \
        np.repeat(np.vectorize(oracle.e4m3_value)(sfs), 16, axis=1) * S
    x = synth.bf16_bits(xv.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(x).astype(np.float64), xv)  # exactly BF16
    a = oracle.forward(x, wr, ex, wl.k, oracle.W4A16, want=("g", "u"))
    b = oracle.forward(x, wr, ex, wl.k, oracle.W4A4, want=("g", "u", "xq_codes", "xq_scales"))
    assert np.array_equal(a["g"], b["g"]) and np.array_equal(a["u"], b["u"])
    qc, qs = oracle.quantize_nvfp4(synth.bf16_to_f32(x), S)
    assert np.array_equal(qs, b["xq_scales"]) and np.array_equal(qc, b["xq_codes"])


def test_forward_w4a4_h_codes_are_q_of_h(tiny):
    wl, x, wr, ex = tiny
    res = oracle.forward(x, wr, ex, wl.k, oracle.W4A4,
                         want=("h", "hq_codes", "hq_scales", "idx", "counts", "h_amb_elem"))
    offs = np.concatenate([[0], np.cumsum(res["counts"])])
    for s in range(wl.T * wl.k):
        e = int(np.searchsorted(offs, s, side="right") - 1)
        c, sc = oracle.quantize_nvfp4(res["h"][s][None, :].astype(np.float32),
                                      float(ex.in_scale[e, 2]))
        assert np.array_equal(c[0], res["hq_codes"][s]) and np.array_equal(sc[0],
                                                                          res["hq_scales"][s])
    assert np.all(res["h_amb_elem"] >= 0)


# ------------------------------------------------------------------ W4A4 h ambiguity window
# The oracle flags the W4A4 h quantiser's decisions that an FP32 evaluation of h could take the
# other way (values within eps * block amax of a rounding boundary) and states how far each such
# flip moves the expert's output. The expected values below are written independently: the
# quantiser's steps in numpy float32 with the brute-force encoders of this file, and the windows
# as closed FP64 intervals around the formats' rounding midpoints.
_E2M1_MAGS = [abs(_e2m1_closed(c)) for c in range(8)]
_E2M1_MIDS = [(_E2M1_MAGS[i] + _E2M1_MAGS[i + 1]) / 2 for i in range(7)]
_E4M3_MAGS = [_e4m3_closed(b) for b in range(0x7F)]
_E4M3_MIDS = [(_E4M3_MAGS[b] + _E4M3_MAGS[b + 1]) / 2 for b in range(0x7E)]
_AMB_EPS = 2.0 ** -14


def _e2m1_brute(v):
    c = _nearest_brute(_E2M1_MAGS, min(abs(v), 6.0), list(range(8)))
    return c | (8 if math.copysign(1, v) < 0 else 0)


def _q_block_ref(v, S, sf=None):
    """The quantiser's steps in numpy float32 (sf given: with that scale instead of its own)."""
    v = np.asarray(v, np.float32)
    S = np.float32(S)
    inv6S = np.float32(1) / (np.float32(6) * S)
    a = np.float32(np.abs(v).max())
    t = a * inv6S
    if sf is None:
        sf = 0x7E if t >= 448 else _nearest_brute(_E4M3_MAGS, float(t), list(range(0x7F)))
    if _E4M3_MAGS[sf] == 0:
        return a, t, sf, np.float32(0), [0] * 16
    r = np.float32(1) / (np.float32(_E4M3_MAGS[sf]) * S)
    return a, t, sf, r, [_e2m1_brute(float(v[i] * r)) for i in range(16)]


def _dec(codes, sf, S):
    return np.array([_e2m1_closed(c) for c in codes]) * _E4M3_MAGS[sf] * float(np.float32(S))


def _amb_ref(v, S, eps, cn):
    a, t, sf, r, codes = _q_block_ref(v, S)
    dec = _dec(codes, sf, S)
    elem = np.zeros(16)
    if r != 0:
        unit = _E4M3_MAGS[sf] * float(np.float32(S))
        win = eps * float(a) * float(r)
        for i in range(16):
            xs = abs(float(np.float32(v[i]) * r))
            for j, m in enumerate(_E2M1_MIDS):
                if xs - win <= m <= xs + win:
                    elem[i] = (_E2M1_MAGS[j + 1] - _E2M1_MAGS[j]) * unit * cn[i]
    block = 0.0
    for b, m in enumerate(_E4M3_MIDS):
        if float(t) * (1 - eps) <= m <= float(t) * (1 + eps):
            alt = b if sf == b + 1 else b + 1
            _, _, _, _, ac = _q_block_ref(v, S, sf=alt)
            block = float(np.sum(np.abs(_dec(ac, alt, S) - dec) * cn))
    return elem, block


def _near(m, f, win):
    """A scaled value at signed distance f * win from the midpoint m."""
    return m + f * win


def test_h_ambiguity_constructed_elements():
    # S = 2^-8 and a block amax of 6 * S give the scale 1.0 (0x38) and r = 256 exactly, so an
    # element's scaled value is v * 256 and the element window is eps * 6 in scaled units
    S = 2.0 ** -8
    win = _AMB_EPS * 6.0
    cn = np.linspace(1.0, 2.5, 16)          # distinct column norms: a wrong index shows
    scaled = [6.0,                           # the amax (never flagged: no boundary above 5)
              0.75, 2.5,                     # exactly on midpoints (ties go to even)
              _near(1.25, 0.6, win), _near(1.75, -0.6, win), _near(3.5, 0.3, win),
              _near(5.0, -0.8, win),         # inside the window, on either side
              _near(0.75, 1.6, win), _near(1.25, -2.0, win), _near(3.5, 4.0, win),
              1.0, 3.0, 0.0,                 # representable, far from every boundary
              -_near(0.25, 0.5, win),        # negative, inside the window of 0.25
              -_near(5.0, 1.5, win),         # negative, outside
              _near(0.25, -0.9, win)]
    v = np.array(scaled, np.float32) / np.float32(256)
    assert np.array_equal(v * np.float32(256), np.array(scaled, np.float32))
    elem, block = oracle.h_ambiguity(v, S, _AMB_EPS, cn)
    ref_e, ref_b = _amb_ref(v, S, _AMB_EPS, cn)
    flagged = {1, 2, 3, 4, 5, 6, 13, 15}
    assert set(np.nonzero(ref_e)[0].tolist()) == flagged
    np.testing.assert_allclose(elem, ref_e, rtol=1e-12, atol=0)
    assert block == 0.0 and ref_b == 0.0
    # closed forms of a few: |dec(alt) - dec(code)| * dec(sf) * S * colnorm
    assert elem[1] == pytest.approx(0.5 * S * cn[1], rel=1e-12)    # 0.5 <-> 1.0
    assert elem[2] == pytest.approx(1.0 * S * cn[2], rel=1e-12)    # 2 <-> 3
    assert elem[6] == pytest.approx(2.0 * S * cn[6], rel=1e-12)    # 4 <-> 6
    assert elem[13] == pytest.approx(0.5 * S * cn[13], rel=1e-12)  # -0 <-> -0.5


def test_h_ambiguity_constructed_block_scales():
    S = 2.0 ** -8
    cn = np.linspace(0.5, 3.0, 16)
    rng = np.random.default_rng(51)
    inv6S = np.float32(1) / (np.float32(6) * np.float32(S))
    for m, f, want in ((1.0625, 0.0, True), (1.0625, 0.5, True), (1.0625, -0.6, True),
                       (1.0625, 3.0, False), (1.0625, -2.5, False), (27.0 / 128, 0.4, True),
                       (100.0, -0.7, True), (100.0, 1.3, False)):
        t_want = m * (1 + f * _AMB_EPS)
        a = np.float32(t_want * 6.0 * S)
        rest = (rng.uniform(-1, 1, 15) * float(a)).astype(np.float32)
        v = np.concatenate([[a], rest]).astype(np.float32)
        t = float(np.float32(a) * inv6S)
        assert abs(t / t_want - 1) < 1e-6
        elem, block = oracle.h_ambiguity(v, S, _AMB_EPS, cn)
        ref_e, ref_b = _amb_ref(v, S, _AMB_EPS, cn)
        assert (ref_b > 0) == want, (m, f)
        assert block == pytest.approx(ref_b, rel=1e-12, abs=0), (m, f)
        np.testing.assert_allclose(elem, ref_e, rtol=1e-12, atol=0)


def test_h_ambiguity_random_blocks_near_boundaries():
    rng = np.random.default_rng(52)
    for it in range(300):
        S = float(np.float32(np.exp(rng.uniform(-9, -2))))
        v = (rng.standard_normal(16) * np.exp(rng.uniform(-2, 2))).astype(np.float32)
        a, t, sf, r, _ = _q_block_ref(v, S)
        if r == 0:
            continue
        win = _AMB_EPS * float(a) * float(r)
        amax_i = int(np.argmax(np.abs(v)))
        for i in range(16):   # move some elements next to an E2M1 midpoint (the amax stays)
            if i != amax_i and rng.random() < 0.5:
                f = rng.uniform(-2.5, 2.5)
                if 0.9 < abs(f) < 1.1:
                    f = 0.5 * np.sign(f)
                m = _E2M1_MIDS[int(rng.integers(0, 7))]
                v[i] = np.float32(np.sign(rng.standard_normal()) * _near(m, f, win) / float(r))
        cn = rng.uniform(0.1, 4.0, 16)
        elem, block = oracle.h_ambiguity(v, S, _AMB_EPS, cn)
        ref_e, ref_b = _amb_ref(v, S, _AMB_EPS, cn)
        np.testing.assert_allclose(elem, ref_e, rtol=1e-12, atol=0, err_msg=str(it))
        assert block == pytest.approx(ref_b, rel=1e-12, abs=0), it


def test_h_ambiguity_flags_exactly_the_codes_a_perturbation_can_change():
    # brute force: move one element by every delta on a fine grid of [-eps*a, eps*a] and
    # re-quantise the block with the quantiser; its code changes for some delta exactly when
    # the oracle flags it (elements placed off the window's edges, so the grid decides)
    S = 2.0 ** -8
    win = _AMB_EPS * 6.0
    cn = np.ones(16)
    rng = np.random.default_rng(53)
    for it in range(40):
        scaled = [6.0] + [float(_near(_E2M1_MIDS[int(rng.integers(0, 7))],
                                      rng.choice([-1, 1]) * rng.choice([0.0, 0.3, 0.7, 1.4, 2.5]),
                                      win)) * float(rng.choice([-1, 1])) for _ in range(15)]
        v = np.array(scaled, np.float32) / np.float32(256)
        elem, _ = oracle.h_ambiguity(v, S, _AMB_EPS, cn)
        a = float(np.abs(v).max())
        c0, s0 = oracle.quantize_nvfp4(v[None, :], S)
        for i in range(1, 16):
            changed = False
            for d in np.linspace(-_AMB_EPS * a, _AMB_EPS * a, 201):
                w = v.copy()
                w[i] = np.float32(float(v[i]) + d)
                c, s = oracle.quantize_nvfp4(w[None, :], S)
                assert s[0, 0] == s0[0, 0]
                ci = (c[0, i // 2] >> (4 * (i % 2))) & 0xF
                c0i = (c0[0, i // 2] >> (4 * (i % 2))) & 0xF
                if (ci & 7) != (c0i & 7):       # a change of magnitude (not only -0 / +0)
                    changed = True
                    break
            assert changed == (elem[i] > 0), (it, i, scaled[i])


def test_forward_h_ambiguity_is_the_block_function(tiny):
    # the forward pass reports, for every slot and block, the block function's values with the
    # expert's down-matrix column norms
    wl, x, wr, ex = tiny
    res = oracle.forward(x, wr, ex, wl.k, oracle.W4A4,
                         want=("h", "idx", "counts", "h_amb_elem", "h_amb_block"))
    offs = np.concatenate([[0], np.cumsum(res["counts"])])
    for s in range(wl.T * wl.k):
        e = int(np.searchsorted(offs, s, side="right") - 1)
        Wd = oracle.dequantize_nvfp4(ex.down[e][0], ex.down[e][1], float(ex.mult[e, 2]))
        cn = np.sqrt((Wd ** 2).sum(axis=0))
        hf = res["h"][s].astype(np.float32)
        for b in range(wl.I // 16):
            ref_e, ref_b = _amb_ref(hf[b * 16:(b + 1) * 16], float(ex.in_scale[e, 2]),
                                    _AMB_EPS, cn[b * 16:(b + 1) * 16])
            np.testing.assert_allclose(res["h_amb_elem"][s, b * 16:(b + 1) * 16], ref_e,
                                       rtol=1e-9, atol=0)
            assert res["h_amb_block"][s, b] == pytest.approx(ref_b, rel=1e-9, abs=0)


# ------------------------------------------------------------------ W4A8 activations
def _e4m3_signed_brute(v):
    """Nearest E4M3 byte of a float (ties to the even byte, saturating at 448), sign kept."""
    a = abs(v)
    b = 0x7E if a >= 448 else _nearest_brute(_E4M3_MAGS, a, list(range(0x7F)))
    return b | (0x80 if math.copysign(1, v) < 0 else 0)


def test_a8_quantizer_matches_numpy_float32_and_brute_force():
    rng = np.random.default_rng(61)
    for _ in range(40):
        S = np.float32(np.exp(rng.uniform(-10, 0)))
        S8 = np.float32(6) * S
        r8 = np.float32(1) / S8
        v = (rng.standard_normal(200) * np.exp(rng.uniform(-6, 6, 200)) * 100 * S8).astype(
            np.float32)
        v[:4] = [0.0, -0.0, -1e-30, 1e30]
        # scaled values on E4M3 midpoints and their neighbours
        mids = np.array(_E4M3_MIDS[::9], np.float32)
        v[4:4 + len(mids)] = (mids / r8).astype(np.float32)
        got = oracle.quantize_a8(v, float(S))
        for i in range(len(v)):
            assert got[i] == _e4m3_signed_brute(float(v[i] * r8)), (float(v[i]), float(S))


def test_a8_quantizer_round_trip_and_saturation():
    rng = np.random.default_rng(62)
    S = 2.0 ** -9 / 6          # S8 = 2^-9 exactly: dec(q) * S8 is exact in float32
    S8 = np.float32(6) * np.float32(S)
    assert S8 == np.float32(2.0 ** -9)
    codes = rng.integers(0, 256, 2000)
    codes = codes[(codes & 0x7F) != 0x7F]                       # no NaN
    v = np.array([_e4m3_closed(int(c)) for c in codes], np.float64) * float(S8)
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)
    got = oracle.quantize_a8(v.astype(np.float32), S)
    assert np.array_equal(got, codes.astype(np.uint8))
    big = oracle.quantize_a8(np.array([1e9, -1e9, 500 * float(S8)], np.float32), S)
    assert list(big) == [0x7E, 0xFE, 0x7E]


def test_forward_w4a8_equals_w4a16_before_h_on_representable_x(tiny):
    wl, _, wr, ex0 = tiny
    rng = np.random.default_rng(63)
    S = 2.0 ** -7 / 6          # S8 = 2^-7
    ex = oracle.ExpertSet(wl.E, wl.H, wl.I)
    for e in range(wl.E):
        ex.set(e, ex0.gate[e], ex0.up[e], ex0.down[e], ex0.mult[e], (S, S, ex0.in_scale[e, 2]))
    codes = rng.integers(0, 256, (wl.T, wl.H))
    codes[(codes & 0x7F) == 0x7F] = 0x3C
    xv = np.vectorize(_e4m3_closed)(codes) * 2.0 ** -7
    x = synth.bf16_bits(xv.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(x).astype(np.float64), xv)   # exactly BF16
    a = oracle.forward(x, wr, ex, wl.k, oracle.W4A16, want=("g", "u"))
    b = oracle.forward(x, wr, ex, wl.k, oracle.W4A8, want=("g", "u", "xq_codes"))
    assert np.array_equal(a["g"], b["g"]) and np.array_equal(a["u"], b["u"])
    assert np.array_equal(b["xq_codes"], oracle.quantize_a8(synth.bf16_to_f32(x), S))


def test_forward_w4a8_h_codes_and_numpy_pipeline(tiny):
    wl, x, wr, ex = tiny
    res = oracle.forward(x, wr, ex, wl.k, oracle.W4A8,
                         want=("h", "g", "u", "hq_codes", "counts", "y", "out64", "idx", "w",
                               "slot_of", "h_amb_elem", "h_amb_block"))
    offs = np.concatenate([[0], np.cumsum(res["counts"])])
    xf = synth.bf16_to_f32(x)
    for s in range(wl.T * wl.k):
        e = int(np.searchsorted(offs, s, side="right") - 1)
        t = [tt for tt in range(wl.T) for j in range(wl.k) if res["slot_of"][tt, j] == s][0]
        Sg, Su, Sd = (float(ex.in_scale[e, i]) for i in range(3))
        # the activations: E4M3 under each matrix's scale, decoded (numpy float32 steps)
        dq = lambda v, S_: np.array([_e4m3_closed(int(c)) for c in oracle.quantize_a8(v, S_)]) \
            * float(np.float32(6) * np.float32(S_))
        Wg = oracle.dequantize_nvfp4(ex.gate[e][0], ex.gate[e][1], float(ex.mult[e, 0]))
        Wu = oracle.dequantize_nvfp4(ex.up[e][0], ex.up[e][1], float(ex.mult[e, 1]))
        Wd = oracle.dequantize_nvfp4(ex.down[e][0], ex.down[e][1], float(ex.mult[e, 2]))
        g = Wg @ dq(xf[t], Sg)
        u = Wu @ dq(xf[t], Su)
        np.testing.assert_allclose(res["g"][s], g, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(res["u"][s], u, rtol=1e-12, atol=1e-14)
        hq = oracle.quantize_a8(res["h"][s].astype(np.float32), Sd)
        assert np.array_equal(hq, res["hq_codes"][s])
        y = Wd @ (np.array([_e4m3_closed(int(c)) for c in hq]) *
                  float(np.float32(6) * np.float32(Sd)))
        yb = synth.bf16_to_f32(synth.bf16_bits(y.astype(np.float64).astype(np.float32)))
        np.testing.assert_allclose(res["y"][s], yb, rtol=2 ** -8, atol=1e-12)
    assert np.all(res["h_amb_block"] == 0)


def _amb8_ref(v, S, eps, cn):
    """Independent window test: element i is flagged when a rounding midpoint lies in the closed
    interval of scaled values it could take; its allowance is the largest move of the nearest
    E4M3 value over that interval (at the interval's ends), times S8 and the column norm."""
    v = np.asarray(v, np.float32)
    S8 = np.float32(6) * np.float32(S)
    r8 = np.float32(1) / S8
    a = float(np.abs(v).max())
    elem = np.zeros(16)
    win = eps * a * float(r8)
    for i in range(16):
        xs = float(v[i] * r8)
        lo, hi = abs(xs) - win, abs(xs) + win
        if any(lo <= m <= hi for m in _E4M3_MIDS):
            q = _e4m3_closed(_e4m3_signed_brute(xs))
            ends = [_e4m3_closed(_e4m3_signed_brute(xs - win)),
                    _e4m3_closed(_e4m3_signed_brute(xs + win))]
            elem[i] = max(abs(d - q) for d in ends) * float(S8) * cn[i]
    return elem


def test_h8_ambiguity_constructed_and_random():
    rng = np.random.default_rng(64)
    for it in range(200):
        S = float(np.float32(np.exp(rng.uniform(-9, -3))))
        r8 = np.float32(1) / (np.float32(6) * np.float32(S))
        v = (rng.standard_normal(16) * 50 / r8).astype(np.float32)
        a = float(np.abs(v).max())
        win = _AMB_EPS * a * float(r8)
        for i in range(16):
            if rng.random() < 0.5 and abs(v[i]) < a * 0.9:
                m = _E4M3_MIDS[int(rng.integers(0, 0x7E))]
                f = rng.uniform(-2.5, 2.5)
                if 0.9 < abs(f) < 1.1:
                    f = 0.4
                if m + f * win < a * float(r8) * 0.95:
                    v[i] = np.float32(np.sign(rng.standard_normal()) * (m + f * win) / float(r8))
        cn = rng.uniform(0.1, 4.0, 16)
        got = oracle.h8_ambiguity(v, S, _AMB_EPS, cn)
        np.testing.assert_allclose(got, _amb8_ref(v, S, _AMB_EPS, cn), rtol=1e-12, atol=0,
                                   err_msg=str(it))
    # an element exactly on a midpoint (1.0625 between 0x38 and 0x39 in scaled units) is flagged
    S = 2.0 ** -8 / 6
    v = np.zeros(16, np.float32)
    v[0] = np.float32(104.0 * 2.0 ** -8)     # the block amax, an E4M3 value (0x6D)
    v[1] = np.float32(1.0625 * 2.0 ** -8)
    got = oracle.h8_ambiguity(v, S, _AMB_EPS, np.ones(16))
    assert got[1] == pytest.approx(0.125 * 2.0 ** -8, rel=1e-12) and got[0] == 0


def test_synth_streams_are_deterministic_and_independent():
    a = synth.expert_weight(0, 3, 7, "gate", 64, 32)
    b = synth.expert_weight(0, 3, 7, "gate", 64, 32)
    c = synth.expert_weight(0, 3, 8, "gate", 64, 32)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert synth.activations(0, 0, 4, 64).shape == (4, 64)


# ------------------------------------------------------------------ shared expert
def _exact_bf16_expert(seed, H, I, S=2.0 ** -12):
    """An NVFP4 expert quantised with a power-of-two multiplier S, so that every dequantised
    weight (code * E4M3 scale * S: at most 6 significant bits) is exactly a BF16 value; returns
    the NVFP4 matrices and the BF16 bit patterns of the dequantised gate, up and down."""
    mats, bf = [], []
    for which in ("gate", "up", "down"):
        w = synth.bf16_to_f32(synth.expert_weight(seed, 0, 0, which, H, I))
        c, s = oracle.quantize_nvfp4(w, S)
        d = oracle.dequantize_nvfp4(c, s, S)
        b = synth.bf16_bits(d.astype(np.float32))
        assert np.array_equal(synth.bf16_to_f32(b).astype(np.float64), d)   # exactly BF16
        mats.append((c, s))
        bf.append(b)
    return mats, bf


def test_shared_expert_equals_routed_expert_with_the_same_weights():
    T, H, E, k, I = 5, 256, 4, 2, 64
    x = synth.activations(41, 0, T, H)
    wr = synth.router_weight(41, 0, E, H)
    (g, u, d), (gb, ub, db) = _exact_bf16_expert(41, H, I)
    ex = oracle.ExpertSet(E, H, I)
    S = 2.0 ** -12
    for e in range(E):
        ex.set(e, g, u, d, (S, S, S))
    routed = oracle.forward(x, wr, ex, k, oracle.W4A16, want=("y", "h_bf16", "slot_of"))
    gv = synth.shared_expert_weights(41, 0, H, I)[2]
    sh = oracle.shared_expert(x, oracle.SharedExpert(np.vstack([gb, ub]), db, gv))
    ys_b = np.array([[oracle.double_to_bf16(v) for v in row] for row in sh["ys"]], np.uint16)
    hs_b = np.array([[oracle.double_to_bf16(v) for v in row] for row in sh["h64"]], np.uint16)
    assert np.array_equal(hs_b, sh["hs_bf16"])
    # Ys is the BF16 rounding of the FP64 down product, like a routed expert's Y
    assert np.array_equal(ys_b, np.array([[oracle.double_to_bf16(v) for v in row]
                                          for row in sh["ys64"]], np.uint16))
    assert np.array_equal(synth.bf16_to_f32(ys_b).astype(np.float64), sh["ys"])
    for t in range(T):
        for j in range(k):
            s = routed["slot_of"][t, j]
            # the routed Y is the BF16 rounding of the same FP64 down product
            assert np.array_equal(synth.bf16_bits(routed["y"][s].astype(np.float32)), ys_b[t])
            assert np.array_equal(routed["h_bf16"][s], sh["hs_bf16"][t])
    # gate and up rows swapped: a different expert (SiLU is not symmetric in g and u)
    sw = oracle.shared_expert(x, oracle.SharedExpert(np.vstack([ub, gb]), db, gv))
    assert not np.array_equal(sw["ys"], sh["ys"])


def test_shared_expert_matches_numpy_float64_pipeline():
    T, H, Is = 3, 128, 64
    x = synth.activations(42, 0, T, H)
    gu, dn, gv = synth.shared_expert_weights(42, 0, H, Is)
    sh = oracle.shared_expert(x, oracle.SharedExpert(gu, dn, gv))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    W = synth.bf16_to_f32(gu).astype(np.float64)
    Wd = synth.bf16_to_f32(dn).astype(np.float64)
    g = xf @ W[:Is].T
    u = xf @ W[Is:].T
    h = g * (1 / (1 + np.exp(-g))) * u
    np.testing.assert_allclose(sh["h64"], h, rtol=1e-12, atol=1e-15)
    hb = np.array([[oracle.double_to_bf16(v) for v in row] for row in h], np.uint16)
    assert np.array_equal(hb, sh["hs_bf16"])
    y = synth.bf16_to_f32(hb).astype(np.float64) @ Wd.T
    np.testing.assert_allclose(sh["ys64"], y, rtol=1e-12, atol=1e-15)
    yb = np.array([[oracle.double_to_bf16(v) for v in row] for row in sh["ys64"]], np.uint16)
    assert np.array_equal(synth.bf16_to_f32(yb).astype(np.float64), sh["ys"])


def test_shared_forward_adds_the_rounded_ys(tiny):
    # out64 = (the routed sum) + sigma_t * BF16(Ys), the shared term added after the routed ones
    wl, x, wr, ex = tiny
    sh = oracle.SharedExpert(*synth.shared_expert_weights(46, 0, wl.H, wl.I))
    a = oracle.forward(x, wr, ex, wl.k, oracle.W4A16)
    b = oracle.forward(x, wr, ex, wl.k, oracle.W4A16, shared=sh)
    assert not np.array_equal(b["ys"], b["ys64"])          # the rounding changed something
    for t in range(wl.T):
        assert np.array_equal(b["out64"][t], a["out64"][t] + b["sigma"][t] * b["ys"][t])
    ob = np.array([[oracle.double_to_bf16(v) for v in row] for row in b["out64"]], np.uint16)
    assert np.array_equal(ob, b["out_bf16"])


def test_shared_gate_is_the_logistic_function():
    from scipy.special import expit
    T, H, Is = 6, 128, 64
    x = synth.activations(43, 0, T, H)
    gu, dn, gv = synth.shared_expert_weights(43, 0, H, Is)
    gv = synth.bf16_bits(synth.bf16_to_f32(gv) * np.float32(8.0))   # a spread of gate values
    sh = oracle.shared_expert(x, oracle.SharedExpert(gu, dn, gv))
    a = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(gv).astype(np.float64)
    assert a.min() < -1 and a.max() > 1
    np.testing.assert_allclose(sh["sigma"], expit(a), rtol=1e-12, atol=0)
    zero = oracle.shared_expert(x, oracle.SharedExpert(gu, dn, np.zeros(H, np.uint16)))
    assert np.all(zero["sigma"] == 0.5)


def test_shared_forward_zero_down_is_the_routed_step(tiny):
    wl, x, wr, ex = tiny
    gu, dn, gv = synth.shared_expert_weights(44, 0, wl.H, wl.I)
    sh = oracle.SharedExpert(gu, np.zeros_like(dn), gv)
    for mode in (oracle.W4A16, oracle.W4A4):
        a = oracle.forward(x, wr, ex, wl.k, mode)
        b = oracle.forward(x, wr, ex, wl.k, mode, shared=sh)
        assert np.all(b["ys"] == 0)
        assert np.array_equal(a["out_bf16"], b["out_bf16"])
        assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["out64"], b["out64"])


def test_shared_forward_closed_form_with_k1_and_equal_experts():
    # k = 1 and every routed expert equal to the shared one, the down rows one-hot with weight
    # 1/8, so that Y = Ys exactly (one exact product per row): out = BF16((1 + sigma_t) * Y_t)
    T, H, E, I = 4, 256, 3, 64
    x = synth.activations(45, 0, T, H)
    wr = synth.router_weight(45, 0, E, H)
    (g, u, _), (gb, ub, _) = _exact_bf16_expert(45, H, I)
    cols = np.random.default_rng(45).integers(0, I, H)
    dc = np.zeros((H, I // 2), np.uint8)
    for r in range(H):
        dc[r, cols[r] // 2] |= 2 << (4 * (cols[r] % 2))          # E2M1 code 2 = 1.0
    d = (dc, np.full((H, I // 16), 0x38, np.uint8))               # E4M3 0x38 = 1.0
    S = 2.0 ** -12
    db = np.zeros((H, I), np.uint16)
    db[np.arange(H), cols] = synth.bf16_bits(np.float32([0.125]))[0]
    assert np.array_equal(oracle.dequantize_nvfp4(*d, 0.125),
                          synth.bf16_to_f32(db).astype(np.float64))
    ex = oracle.ExpertSet(E, H, I)
    for e in range(E):
        ex.set(e, g, u, d, (S, S, 0.125))
    for gv in (np.zeros(H, np.uint16), synth.shared_expert_weights(45, 0, H, I)[2]):
        res = oracle.forward(x, wr, ex, 1, oracle.W4A16, want=("out64", "y", "slot_of"),
                             shared=oracle.SharedExpert(np.vstack([gb, ub]), db, gv))
        for t in range(T):
            y = res["y"][res["slot_of"][t, 0]]
            assert np.array_equal(y, res["ys"][t])
            if not gv.any():
                assert res["sigma"][t] == 0.5
                assert np.array_equal(res["out64"][t], 1.5 * y)   # exact: y has 8 bits
            np.testing.assert_allclose(res["out64"][t], (1 + res["sigma"][t]) * y, rtol=1e-15,
                                       atol=0)
            ob = np.array([oracle.double_to_bf16(v) for v in res["out64"][t]], np.uint16)
            assert np.array_equal(ob, res["out_bf16"][t])
