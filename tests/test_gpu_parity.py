"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded
inputs. Rules and tolerances are stated in tests/_gpu_fixtures.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
import nvfp4_mixture_experts_bf16_gb300 as moe
from _gpu_fixtures import (GAMMA_NARROW, GAMMA_WIDE, FullLayer, check_topk, compare_outputs,
                           dev_bf16, gamma, h8_flip_allowance, h_flip_allowance, host_u16,
                           pack_from_experts, slot_map, small_layer, stable_perm, ws_array)

pytestmark = pytest.mark.gpu

ALL = ("out_bf16", "out64", "logits", "abssum", "idx", "w", "counts", "offsets", "perm",
       "slot_of", "h_bf16", "hq_codes", "hq_scales", "h_amb_elem", "h_amb_block", "y",
       "xq_codes", "xq_scales")


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.lib()


def run_and_check(x, wr, ex, pack, k, mode, nthreads=8, tokens=None, shared=None):
    """Run moe_forward (moe_forward_shared when ``shared`` = (gate_up, down, gate) BF16 arrays
    is given) on the GPU and check every stage against the oracle."""
    T, H = x.shape
    E, I = ex.E, ex.I
    S = T * k
    if shared is None:
        ws = moe.new_workspace(moe.moe_workspace_size(pack, T, k, mode))
        out = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, k, mode, ws=ws)
    else:
        Is = shared[0].shape[0] // 2
        ws = moe.new_workspace(moe.moe_workspace_size_shared(pack, T, k, mode, Is))
        out = moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack,
                                     tuple(dev_bf16(a) for a in shared), k, mode, ws=ws)
    launches = moe.moe_last_launch_count()
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    off = moe.moe_workspace_offsets(pack, T, k, mode)
    g_idx = ws_array(ws, off["idx"], S * 4, np.int32).reshape(T, k)
    g_w = ws_array(ws, off["w"], S * 4, np.float32).reshape(T, k)
    g_counts = ws_array(ws, off["counts"], E * 4, np.int32)
    g_offsets = ws_array(ws, off["offsets"], (E + 1) * 4, np.int32)
    g_perm = ws_array(ws, off["perm"], S * 4, np.int32)
    g_slot_of = ws_array(ws, off["slot_of"], S * 4, np.int32).reshape(T, k)
    ref = oracle.forward(x, wr, ex, k, mode, nthreads=nthreads, want=ALL,
                         shared=None if shared is None else oracle.SharedExpert(*shared))
    sh_allow = {} if shared is None else check_shared(ws, pack, x, shared, ref, k, mode)

    differ = check_topk(g_idx, g_w, ref, GAMMA_NARROW if T <= 8 else GAMMA_WIDE)
    c, o, p = stable_perm(g_idx, E)
    assert np.array_equal(g_counts, c) and np.array_equal(g_offsets, o)
    assert np.array_equal(g_perm, p)
    if not differ:
        assert np.array_equal(g_perm, ref["perm"]) and np.array_equal(g_counts, ref["counts"])
    for t in range(T):
        for j in range(k):
            s = g_slot_of[t, j]
            assert g_perm[s] == t and g_offsets[g_idx[t, j]] <= s < g_offsets[g_idx[t, j] + 1]

    if mode == 1:
        assert np.array_equal(ws_array(ws, off["x_codes"], T * H // 2, np.uint8).reshape(T, -1),
                              ref["xq_codes"])
        assert np.array_equal(ws_array(ws, off["x_scales"], T * H // 16, np.uint8).reshape(T, -1),
                              ref["xq_scales"])
    if mode == 2:
        assert np.array_equal(ws_array(ws, off["x_codes"], T * H, np.uint8).reshape(T, H),
                              ref["xq_codes"])
    gm = slot_map(g_perm, g_offsets)
    rm = slot_map(ref["perm"], ref["offsets"])
    allowance = dict(sh_allow)
    flips = 0
    if mode == 0:
        gh = synth.bf16_to_f32(ws_array(ws, off["h_bf16"], S * I * 2, np.uint16).reshape(S, I))
        rh = synth.bf16_to_f32(ref["h_bf16"])
        gy = synth.bf16_to_f32(ws_array(ws, off["y"], S * H * 2, np.uint16).reshape(S, H))
    elif mode == 1:
        gq = ws_array(ws, off["h_codes"], S * I // 2, np.uint8).reshape(S, I // 2)
        gsf = ws_array(ws, off["h_scales"], S * I // 16, np.uint8).reshape(S, I // 16)
    else:
        gq8 = ws_array(ws, off["h_codes"], S * I, np.uint8).reshape(S, I)
    for t in range(T):
        if t in differ:
            continue
        for j in range(k):
            e = int(g_idx[t, j])
            gs, rs = gm[(t, e)], rm[(t, e)]
            if mode == 0:
                a, b = gh[gs].astype(np.float64), rh[rs].astype(np.float64)
                scale = np.sqrt(np.mean(b * b)) + 1e-30
                # at most one BF16 ulp (<= 2^-7 of the larger magnitude) where the FP32 h and
                # the FP64 h round to different neighbours
                assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b))
                              + 1e-5 * scale), (t, j, np.flatnonzero(np.abs(a - b) > 2.0 ** -7 *
                                                np.maximum(np.abs(a), np.abs(b)) + 1e-5 * scale))
                ya, yb = gy[gs].astype(np.float64), ref["y"][rs]
                assert np.linalg.norm(ya - yb) <= 2e-3 * np.linalg.norm(yb) + 1e-30, (t, j)
            else:
                if mode == 1:
                    a, f = h_flip_allowance(gq[gs], gsf[gs], ref, rs, I)
                else:
                    a, f = h8_flip_allowance(gq8[gs], ref, rs)
                allowance[t] = allowance.get(t, 0.0) + float(g_w[t, j]) * a
                flips += f
    toks = [t for t in range(T) if t not in differ] if tokens is None else tokens
    worst = compare_outputs(host_u16(out), ref, mode, toks, allowance)
    return dict(out=out, ws=ws, differ=differ, flips=flips, worst=worst, ref=ref, g_idx=g_idx,
                launches=launches)


def check_shared(ws, pack, x, shared, ref, k, mode):
    """The shared expert's intermediates against the oracle; returns, per token, the output
    allowance of its accepted h roundings.

    The gate: within the FP32 bound of its dot product. h: equal to the oracle's BF16 h, or
    else between the BF16 roundings of h64 - win and h64 + win (rounding is monotonic), h64
    being the oracle's unrounded h and win the FP32 error bound of the GPU's h:
    |u| * 1.1 * dg + |SiLU(g)| * du + 8 ulp(h), with dg, du = gamma_n * sum|x * w| the FP32
    accumulation bounds of g and u (n as for the router). Each accepted difference widens the
    token's Ys bound by |dh| * ||Wd[:, i]||_2, its exact effect on Ys (triangle inequality). Ys
    before its BF16 rounding (FP32, as the workspace holds it): per token within 1e-4 of the
    oracle's unrounded Ys norm plus that allowance. Both sides round Ys to BF16 before the
    combine; where a validated Ys and the oracle's straddle a BF16 rounding boundary the two
    roundings differ by one BF16 step, so the token's output allowance is sigma_t times the L2
    distance of the two rounded Ys (which also carries the accepted h differences)."""
    T, H = x.shape
    Is = shared[0].shape[0] // 2
    so = moe.moe_workspace_offsets_shared(pack, T, k, mode, Is)
    return check_shared_arrays(
        x, shared, ref, ws_array(ws, so["sigma"], T * 4, np.float32),
        ws_array(ws, so["h"], T * Is * 2, np.uint16).reshape(T, Is),
        ws_array(ws, so["y"], T * H * 4, np.float32).reshape(T, H))


def check_shared_arrays(x, shared, ref, sig, gh_bits, gy):
    """check_shared on host arrays: sigma [T] float32, h [T, Is] BF16 bits, Ys [T, H] float32."""
    T, H = x.shape
    gu, dn, gv = shared
    Is = gu.shape[0] // 2
    sig = np.asarray(sig, np.float64)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    xa = np.abs(xf)
    bound = 0.25 * gamma(GAMMA_WIDE) * (xa @ np.abs(synth.bf16_to_f32(gv).astype(np.float64)))
    assert np.all(np.abs(sig - ref["sigma"]) <= bound + 1e-6), np.abs(sig - ref["sigma"]).max()
    gh = synth.bf16_to_f32(gh_bits).astype(np.float64)
    rh = synth.bf16_to_f32(ref["hs_bf16"]).astype(np.float64)
    diff = np.nonzero(gh != rh)
    allow = np.zeros(T)
    if len(diff[0]):
        W = synth.bf16_to_f32(gu).astype(np.float64)
        wg, wu = W[:Is], W[Is:]
        wcol = np.linalg.norm(synth.bf16_to_f32(dn).astype(np.float64), axis=0)  # ||Wd[:, i]||
        for t, i in zip(*diff):
            g, u = xf[t] @ wg[i], xf[t] @ wu[i]
            dg = gamma(GAMMA_WIDE) * (xa[t] @ np.abs(wg[i]))
            du = gamma(GAMMA_WIDE) * (xa[t] @ np.abs(wu[i]))
            win = abs(u) * 1.1 * dg + abs(g / (1 + np.exp(-g))) * du + 8 * 2.0 ** -24 * abs(g * u)
            h64 = ref["hs64"][t, i]
            lo = synth.bf16_to_f32(np.uint16(oracle.double_to_bf16(h64 - win)))
            hi = synth.bf16_to_f32(np.uint16(oracle.double_to_bf16(h64 + win)))
            assert lo <= gh[t, i] <= hi, ("h outside the rounding of its error interval", t, i,
                                          gh[t, i], rh[t, i], h64, win)
            allow[t] += abs(gh[t, i] - rh[t, i]) * wcol[i]
    gy = np.asarray(gy, np.float32)
    gyb = synth.bf16_to_f32(synth.bf16_bits(gy)).astype(np.float64)   # RNE, as the combines do
    out_allow = {}
    for t in range(T):
        ny = np.linalg.norm(ref["ys64"][t])
        assert np.linalg.norm(gy[t].astype(np.float64) - ref["ys64"][t]) <= \
            1e-4 * ny + allow[t] * (1 + 1e-6) + 1e-30, t
        d = float(np.linalg.norm(gyb[t] - ref["ys"][t]))
        if d > 0:
            out_allow[t] = float(ref["sigma"][t]) * d
    return out_allow


# ------------------------------------------------------------------ quantiser
def _q_case(rows, cols, S, rng):
    v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-4, 4, (rows, 1)))
    v[0, :16] = 0.0                       # a zero block
    v[1, :16] = 1e30                      # saturating block
    v[1, 3] = -1e30
    return synth.bf16_bits(v.astype(np.float32))


def test_quantizer_bit_exact_random():
    rng = np.random.default_rng(0)
    for S in (1e-3, 0.37, 2.0 ** -9, 5e-6):
        xb = _q_case(96, 1024, S, rng)
        gc, gs = moe.moe_quantize_act_nvfp4(dev_bf16(xb), S)
        rc, rs = oracle.quantize_nvfp4(synth.bf16_to_f32(xb), S)
        assert np.array_equal(gs.cpu().numpy(), rs), S
        assert np.array_equal(gc.cpu().numpy(), rc), S


def test_quantizer_bit_exact_on_rounding_ties():
    # S and the block scale are powers of two, so v * r lands exactly on E2M1 midpoints.
    S = 2.0 ** -9
    rows = []
    rng = np.random.default_rng(1)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 6.0, 0.0]
    for k2 in range(-6, 7):
        blk = np.array([6.0] + list(rng.choice(mids, 15)), np.float64) * 2.0 ** k2
        blk *= np.where(rng.random(16) < 0.5, -1, 1)
        rows.append(blk)
    xb = synth.bf16_bits(np.array(rows, np.float32))
    assert np.array_equal(synth.bf16_to_f32(xb), np.array(rows, np.float32))
    gc, gs = moe.moe_quantize_act_nvfp4(dev_bf16(xb), S)
    rc, rs = oracle.quantize_nvfp4(synth.bf16_to_f32(xb), S)
    assert np.array_equal(gs.cpu().numpy(), rs)
    assert np.array_equal(gc.cpu().numpy(), rc)


# ------------------------------------------------------------------ pack
def test_pack_is_bit_preserving():
    x, wr, ex = small_layer(1, 256, 5, 2, 64)
    pack = pack_from_experts(ex)
    for e in range(ex.E):
        for which, m in ((0, ex.gate), (1, ex.up), (2, ex.down)):
            c, s, mult, ins = pack.get_matrix(e, which)
            assert np.array_equal(c, m[e][0]) and np.array_equal(s, m[e][1])
            assert np.float32(mult) == ex.mult[e, which]
            assert np.float32(ins) == ex.in_scale[e, which]
    pack.close()


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("T", [1, 5, 8, 9, 37, 300])
def test_route_topk(T):
    H, E, k = 512, 96, 6
    x = synth.activations(3, 0, T, H, zipf=True)
    wr = synth.router_weight(3, 0, E, H, zipf=True)
    g = moe.moe_route_topk(dev_bf16(x), dev_bf16(wr), k)
    torch.cuda.synchronize()
    ref = oracle.route(x, wr, k, nthreads=8)
    gi = g["idx"].cpu().numpy()
    differ = check_topk(gi, g["w"].cpu().numpy(), ref, GAMMA_NARROW if T <= 8 else GAMMA_WIDE)
    c, o, p = stable_perm(gi, E)
    assert np.array_equal(g["counts"].cpu().numpy(), c)
    assert np.array_equal(g["offsets"].cpu().numpy(), o)
    assert np.array_equal(g["perm"].cpu().numpy(), p)
    if not differ:
        assert np.array_equal(p, ref["perm"])


def test_route_topk_full_size_router():
    for T in (1, 8):
        x = synth.activations(0, 7, T, 4096, zipf=T == 8)
        wr = synth.router_weight(0, 7, 512, 4096, zipf=T == 8)
        g = moe.moe_route_topk(dev_bf16(x), dev_bf16(wr), 10)
        torch.cuda.synchronize()
        ref = oracle.route(x, wr, 10, nthreads=8)
        differ = check_topk(g["idx"].cpu().numpy(), g["w"].cpu().numpy(), ref, GAMMA_NARROW)
        assert not differ


def test_route_ties_go_to_lower_index():
    T, H, E, k = 3, 256, 32, 5
    x = synth.activations(5, 0, T, H)
    wr = np.tile(synth.router_weight(5, 0, 1, H), (E, 1))  # all logits equal
    g = moe.moe_route_topk(dev_bf16(x), dev_bf16(wr), k)
    gi = g["idx"].cpu().numpy()
    assert np.array_equal(gi, np.tile(np.arange(k), (T, 1)))
    assert np.allclose(g["w"].cpu().numpy(), 1.0 / k, rtol=1e-6)


# ------------------------------------------------------------------ forward, small shapes
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_forward_tiny_workload(mode):
    wl = synth.WORKLOADS["tiny"]
    x, wr, ex = small_layer(wl.T, wl.H, wl.E, wl.k, wl.I)
    pack = pack_from_experts(ex)
    r = run_and_check(x, wr, ex, pack, wl.k, mode)
    assert r["worst"] < {0: 2e-3, 1: 5e-3, 2: 5e-3}[mode]
    pack.close()


@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 50, 203])
def test_forward_w4a8_ragged_shapes(T):
    # W4A8 (E4M3 activations): the fused narrow kernel (T <= 8) and the tensor-core f16 path
    H, E, k, I = 1536, 24, 4, 256
    x, wr, ex = small_layer(T, H, E, k, I, zipf=True, seed=12)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, 2)
    pack.close()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 50, 203])
def test_forward_ragged_shapes(T, mode):
    # several row tiles, k-blocks and token groups, with ragged tails
    H, E, k, I = 1536, 24, 4, 192
    x, wr, ex = small_layer(T, H, E, k, I, zipf=True, seed=11)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, mode)
    pack.close()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("T,H,E,k,I", [
    (1, 768, 640, 8, 128),    # more than 512 experts (32 logits per lane), H % 512 != 0
    (2, 768, 640, 8, 128),
    (1, 1024, 64, 1, 128),    # a single expert per token
    (1, 1024, 64, 16, 128),   # 16 experts per token
    (5, 1024, 200, 6, 256),
])
def test_forward_narrow_call_shapes(T, H, E, k, I, mode):
    # the one-launch narrow-call kernel (T <= 8): router dot products on CUDA cores (T <= 2) or
    # tensor cores, the threshold top-k with 16 or 32 logits per lane, one-token groups built in
    # the selecting warp
    x, wr, ex = small_layer(T, H, E, k, I, seed=31 + T + k)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, mode)
    pack.close()


@pytest.mark.parametrize("mode", [1, 0, 2])
def test_forward_multi_tile_experts(mode):
    # every expert receives more than 128 slots: several token tiles per expert on the grouped
    # tensor-core path (W4A4), several 8-token groups on the grouped CUDA-core path (W4A16)
    T, H, E, k, I = 600, 512, 8, 2, 128
    x, wr, ex = small_layer(T, H, E, k, I, seed=21)
    pack = pack_from_experts(ex)
    r = run_and_check(x, wr, ex, pack, k, mode)
    assert np.bincount(r["g_idx"].ravel(), minlength=E).max() > 128
    pack.close()


def test_forward_twice_is_deterministic_and_counters_reset():
    x, wr, ex = small_layer(8, 512, 32, 4, 128, seed=4)
    pack = pack_from_experts(ex)
    ws = moe.new_workspace(moe.moe_workspace_size(pack, 8, 4, 0))
    a = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, 4, 0, ws=ws).clone()
    b = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, 4, 0, ws=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_read_device_status(ws) == 0
    assert int(ws[:4].view(torch.int32).item()) == 0     # router ticket back at zero
    pack.close()


def test_forward_modes_interleaved_on_one_workspace():
    # narrow calls of all three modes (and a wide call) share one workspace: the fused kernel's
    # control words (epoch, CTA counters) must carry over between them, so every output equals
    # the same call's output on a fresh workspace, and a T = 1 and a T = 8 call alternate too
    H, E, k, I = 512, 32, 4, 128
    x8, wr, ex = small_layer(8, H, E, k, I, seed=5)
    pack = pack_from_experts(ex)
    size = max(moe.moe_workspace_size(pack, T, k, m) for T in (1, 8, 40) for m in (0, 1, 2))
    ws = moe.new_workspace(size)
    x40 = small_layer(40, H, E, k, I, seed=5)[0]
    calls = [(8, 0), (8, 1), (1, 2), (8, 2), (40, 1), (1, 0), (8, 1), (1, 1), (8, 0)]
    for T, mode in calls:
        xs = x8[:T] if T <= 8 else x40
        got = moe.moe_forward(dev_bf16(xs), dev_bf16(wr), pack, k, mode, ws=ws).clone()
        fresh = moe.moe_forward(dev_bf16(xs), dev_bf16(wr), pack, k, mode).clone()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), fresh.view(torch.int16)), (T, mode)
        assert moe.moe_read_device_status(ws) == 0, (T, mode)
    pack.close()


def test_forward_identical_experts_equal_one_expert():
    x, wr, ex = small_layer(4, 512, 16, 3, 128, seed=6)
    same = oracle.ExpertSet(ex.E, ex.H, ex.I)
    for e in range(ex.E):
        same.set(e, ex.gate[0], ex.up[0], ex.down[0], ex.mult[0], ex.in_scale[0])
    pack = pack_from_experts(same)
    r = run_and_check(x, wr, same, pack, 3, 0)
    # every slot of a token holds the same Y; the weights sum to 1
    ref = r["ref"]
    for t in range(4):
        y0 = ref["y"][ref["slot_of"][t, 0]]
        assert np.array_equal(synth.bf16_to_f32(ref["out_bf16"][t]).astype(np.float64), y0)
    pack.close()


def test_forward_zero_activations():
    x = np.zeros((3, 512), np.uint16)
    _, wr, ex = small_layer(3, 512, 16, 3, 128, seed=8)
    pack = pack_from_experts(ex)
    for mode in (0, 1):
        out = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, 3, mode)
        torch.cuda.synchronize()
        assert torch.count_nonzero(out.float()).item() == 0
    pack.close()


def test_forward_rejects_bad_arguments():
    x, wr, ex = small_layer(2, 256, 8, 2, 64)
    pack = pack_from_experts(ex)
    xd, wd = dev_bf16(x), dev_bf16(wr)
    with pytest.raises(moe.MoeError):
        moe.moe_forward(xd, wd, pack, 9, 0)            # k > E
    ws = moe.new_workspace(64)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(xd, wd, pack, 2, 0, ws=ws)      # workspace too small
    assert e.value.code == 6
    pack.close()


# ------------------------------------------------------------------ full-size decode
@pytest.mark.parametrize("name", ["decode1", "verify8", "verify8_w4a4", "verify8_w4a8"])
def test_forward_full_size_decode(name):
    wl = synth.WORKLOADS[name]
    lay = FullLayer(0, 0, wl.T, wl.zipf)
    ref_route = oracle.route(lay.x, lay.wr, wl.k, nthreads=8)
    ex = lay.oracle_experts(ref_route["idx"].ravel())
    r = run_and_check(lay.x, lay.wr, ex, lay.pack, wl.k, wl.mode)
    assert not r["differ"]
    lay.close()


# ------------------------------------------------------------------ full-size prefill, sampled
@pytest.mark.parametrize("mode,with_shared", [(1, False), (0, False), (1, True), (2, False)])
def test_forward_prefill_8192_sampled(mode, with_shared):
    wl = synth.WORKLOADS["prefill8192"]
    lay = FullLayer(0, 0, wl.T, wl.zipf)
    T, k = wl.T, wl.k
    shared = synth.shared_expert_weights(0, 0, lay.H, lay.I) if with_shared else None
    if shared is None:
        ws = moe.new_workspace(moe.moe_workspace_size(lay.pack, T, k, mode))
        out = moe.moe_forward(dev_bf16(lay.x), dev_bf16(lay.wr), lay.pack, k, mode, ws=ws)
    else:
        ws = moe.new_workspace(moe.moe_workspace_size_shared(lay.pack, T, k, mode, lay.I))
        out = moe.moe_forward_shared(dev_bf16(lay.x), dev_bf16(lay.wr), lay.pack,
                                     tuple(dev_bf16(a) for a in shared), k, mode, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    off = moe.moe_workspace_offsets(lay.pack, T, k, mode)
    g_idx = ws_array(ws, off["idx"], T * k * 4, np.int32).reshape(T, k)
    g_w = ws_array(ws, off["w"], T * k * 4, np.float32).reshape(T, k)
    ref_route = oracle.route(lay.x, lay.wr, k, nthreads=16)
    differ = check_topk(g_idx, g_w, ref_route, GAMMA_WIDE)
    c, o, p = stable_perm(g_idx, lay.E)
    assert np.array_equal(ws_array(ws, off["perm"], T * k * 4, np.int32), p)
    assert c.max() > 1000  # the Zipf popularity reaches the thousands
    if mode == 1:
        rc, rs = oracle.quantize_nvfp4(synth.bf16_to_f32(lay.x), lay.xs, nthreads=16)
        assert np.array_equal(ws_array(ws, off["x_codes"], T * 2048, np.uint8).reshape(T, -1), rc)
        assert np.array_equal(ws_array(ws, off["x_scales"], T * 256, np.uint8).reshape(T, -1), rs)
    if mode == 2:
        rc = oracle.quantize_a8(synth.bf16_to_f32(lay.x), lay.xs)
        assert np.array_equal(ws_array(ws, off["x_codes"], T * lay.H, np.uint8).reshape(T, -1),
                              rc)
    rng = np.random.default_rng(0)
    sample = [int(t) for t in rng.choice(T, 24, replace=False) if t not in differ]
    sample += [t for t in (0, T - 1) if t not in differ and t not in sample]
    # on purpose: tokens of the two busiest experts (more than 1000 slots, many 128-slot token
    # tiles each): the first, middle and last slots of each, so the last (ragged) token tile of
    # a hot expert is always compared
    g_perm_all = ws_array(ws, off["perm"], T * k * 4, np.int32)
    for e_hot in np.argsort(-c, kind="stable")[:2]:
        for s_ in (o[e_hot], (o[e_hot] + o[e_hot + 1]) // 2, o[e_hot + 1] - 1):
            t = int(g_perm_all[s_])
            if t not in differ and t not in sample:
                sample.append(t)
    ex = lay.oracle_experts(ref_route["idx"][sample].ravel(), nthreads=16)
    ref = oracle.forward(lay.x[sample], lay.wr, ex, k, mode, nthreads=16,
                         want=("out_bf16", "out64", "idx", "perm", "offsets", "hq_codes",
                               "hq_scales", "h_amb_elem", "h_amb_block", "y", "h_bf16"),
                         shared=None if shared is None else oracle.SharedExpert(*shared))
    # every sampled slot's expert output Y (and h in W4A16) against the oracle's
    gm_all = slot_map(g_perm_all, o)
    rm_all = slot_map(ref["perm"], ref["offsets"])
    gy = ws_array(ws, off["y"], T * k * lay.H * 2, np.uint16).reshape(T * k, lay.H)
    if mode == 0:
        gh = ws_array(ws, off["h_bf16"], T * k * lay.I * 2, np.uint16).reshape(T * k, lay.I)
    for i, t in enumerate(sample):
        for j in range(k):
            e = int(g_idx[t, j])
            gs, rs_ = gm_all[(t, e)], rm_all[(i, e)]
            if mode == 0:
                a = synth.bf16_to_f32(gh[gs]).astype(np.float64)
                b = synth.bf16_to_f32(ref["h_bf16"][rs_]).astype(np.float64)
                scale = np.sqrt(np.mean(b * b)) + 1e-30
                assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b))
                              + 1e-5 * scale), (t, j)
                # Y of the slots whose h is the oracle's bit for bit: an accepted one-ulp h
                # difference moves every element of Y, and its BF16 re-rounding amplifies that
                # (those slots stay covered by the h check above and the output bound below)
                if np.array_equal(gh[gs], ref["h_bf16"][rs_]):
                    ya = synth.bf16_to_f32(gy[gs]).astype(np.float64)
                    assert np.linalg.norm(ya - ref["y"][rs_]) <= \
                        2e-3 * np.linalg.norm(ref["y"][rs_]), (t, j)
    allowance = {}
    if mode == 1:
        g_perm = ws_array(ws, off["perm"], T * k * 4, np.int32)
        gm = slot_map(g_perm, o)
        rm = slot_map(ref["perm"], ref["offsets"])
        gq = ws_array(ws, off["h_codes"], T * k * lay.I // 2, np.uint8).reshape(T * k, -1)
        gsf = ws_array(ws, off["h_scales"], T * k * lay.I // 16, np.uint8).reshape(T * k, -1)
        for i, t in enumerate(sample):
            for j in range(k):
                e = int(g_idx[t, j])
                a, _ = h_flip_allowance(gq[gm[(t, e)]], gsf[gm[(t, e)]], ref, rm[(i, e)], lay.I)
                allowance[i] = allowance.get(i, 0.0) + float(g_w[t, j]) * a
    if mode == 2:
        g_perm = ws_array(ws, off["perm"], T * k * 4, np.int32)
        gm = slot_map(g_perm, o)
        rm = slot_map(ref["perm"], ref["offsets"])
        gq8 = ws_array(ws, off["h_codes"], T * k * lay.I, np.uint8).reshape(T * k, -1)
        for i, t in enumerate(sample):
            for j in range(k):
                e = int(g_idx[t, j])
                a, _ = h8_flip_allowance(gq8[gm[(t, e)]], ref, rm[(i, e)])
                allowance[i] = allowance.get(i, 0.0) + float(g_w[t, j]) * a
    got = host_u16(out)[sample]
    compare_outputs(got, ref, mode, list(range(len(sample))), allowance)
    lay.close()


# ------------------------------------------------------------------ shared expert
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 203])
def test_forward_shared_ragged_shapes(T, mode):
    # one or two tokens: the shared expert inside the one-launch routed kernel; three to eight:
    # the two CUDA-core GEMVs then the routed kernel; wide calls: the two tcgen05 BF16 GEMMs
    # with the per-token kernel between them
    H, E, k, I = 1536, 24, 4, 192
    x, wr, ex = small_layer(T, H, E, k, I, zipf=True, seed=11)
    pack = pack_from_experts(ex)
    r = run_and_check(x, wr, ex, pack, k, mode, shared=synth.shared_expert_weights(11, 0, H, I))
    if T <= 2:
        assert r["launches"] == 1
    elif T <= 8:
        assert r["launches"] == 3
    pack.close()


@pytest.mark.parametrize("T,H,E,k,I,Is", [
    (4, 256, 16, 2, 64, 64),      # the tiny workload's shapes, Is = I
    (3, 1024, 64, 6, 128, 640),   # Is > 512: the down rows' units past the register-held ones
    (40, 1024, 64, 6, 128, 640),  # the same through the tensor-core GEMMs (K = 640)
    (2, 4096, 64, 10, 384, 384),  # decode widths (H, I, Is) with 64 experts
    (1, 1024, 64, 6, 128, 640),   # one token, inside the fused kernel, Is > 512
    (1, 4096, 64, 10, 384, 2048),  # one token whose gate/up rows exceed the fused kernel's
                                   # shared memory: the two separate GEMVs instead
])
def test_forward_shared_shapes(T, H, E, k, I, Is):
    x, wr, ex = small_layer(T, H, E, k, I, seed=50 + T)
    pack = pack_from_experts(ex)
    r = run_and_check(x, wr, ex, pack, k, 0, shared=synth.shared_expert_weights(50 + T, 0, H, Is))
    if T <= 2:
        assert r["launches"] == (3 if Is == 2048 else 1)
    pack.close()


@pytest.mark.parametrize("T", [1, 5, 50])
def test_forward_shared_zero_down_is_moe_forward(T):
    # the shared term sigma * BF16(0) leaves the routed sum unchanged: bit-identical outputs
    H, E, k, I = 512, 32, 4, 128
    x, wr, ex = small_layer(T, H, E, k, I, seed=61)
    pack = pack_from_experts(ex)
    gu, dn, gv = synth.shared_expert_weights(61, 0, H, I)
    for mode in (0, 1):
        a = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, k, mode).clone()
        sh = (dev_bf16(gu), dev_bf16(np.zeros_like(dn)), dev_bf16(gv))
        b = moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack, sh, k, mode).clone()
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (T, mode)
    pack.close()


def test_forward_shared_twice_is_deterministic():
    for T in (1, 8, 40):
        x, wr, ex = small_layer(T, 512, 32, 4, 128, seed=62)
        pack = pack_from_experts(ex)
        sh = tuple(dev_bf16(a) for a in synth.shared_expert_weights(62, 0, 512, 128))
        ws = moe.new_workspace(moe.moe_workspace_size_shared(pack, T, 4, 0, 128))
        a = moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack, sh, 4, 0, ws=ws).clone()
        b = moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack, sh, 4, 0, ws=ws).clone()
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert moe.moe_read_device_status(ws) == 0
        pack.close()


def test_forward_shared_rejects_bad_arguments():
    x, wr, ex = small_layer(2, 256, 8, 2, 64)
    pack = pack_from_experts(ex)
    gu, dn, gv = (dev_bf16(a) for a in synth.shared_expert_weights(0, 0, 256, 64))
    with pytest.raises(moe.MoeError):                      # inter % 64 != 0
        moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack, (gu[:100], dn, gv), 2, 0)
    with pytest.raises(moe.MoeError) as e:                  # workspace without the shared part
        moe.moe_forward_shared(dev_bf16(x), dev_bf16(wr), pack, (gu, dn, gv), 2, 0,
                               ws=moe.new_workspace(moe.moe_workspace_size(pack, 2, 2, 0)))
    assert e.value.code == 6
    pack.close()


@pytest.mark.parametrize("name", ["decode1", "verify8_w4a4"])
def test_forward_shared_full_size_decode(name):
    wl = synth.WORKLOADS[name]
    lay = FullLayer(0, 0, wl.T, wl.zipf)
    ref_route = oracle.route(lay.x, lay.wr, wl.k, nthreads=8)
    ex = lay.oracle_experts(ref_route["idx"].ravel())
    r = run_and_check(lay.x, lay.wr, ex, lay.pack, wl.k, wl.mode,
                      shared=synth.shared_expert_weights(0, 0, lay.H, lay.I))
    # decode1 (one token): the shared expert inside the routed kernel; verify8: two GEMVs first
    assert not r["differ"] and r["launches"] == (1 if wl.T <= 2 else 3)
    lay.close()
