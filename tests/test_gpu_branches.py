"""GPU parity of the dispatch branches that the main parity shapes do not reach, and of layers
chained through one workspace.

Branches (each compared with the oracle under the rules of tests/_gpu_fixtures.py):
* the narrow multi-kernel path (router, gate/up, down, combine as four launches), taken when a
  shape does not fit the one-launch narrow kernel: H % 256 != 0, or an activation operand too
  large for one SM's shared memory (T = 8 at H = 8192);
* the wide W4A16 tensor-core path with the down GEMM's h tile re-staged (k_tc16<true>): H % 256
  != 0, or an h tile too large to stay resident (I = 1536);
* the wide grouped mma.sync path: W4A4 with H % 256 != 0, W4A16 with I % 128 != 0;
* the W4A4 down GEMM with the token tile's h resident (several I), and with h restaged per unit
  (an I whose h tile does not fit twice beside two weight tiles);
* the W4A16 / W4A8 resident-h down GEMM (k_tc16_dn) with Y stored in TMA boxes (32- and 16-row
  boxes plus plain stores for a ragged tile's last rows) and, where the h tile leaves no room
  for the staging (I = 512), with plain row stores only;
* W4A4 with unequal gate/up input scales, which the library refuses (MOE_ERR_UNSUPPORTED).

Chained layers: layer l's output is layer l+1's input, every layer with its own router and
experts, all calls queued back to back on one stream and one workspace (programmatic dependent
launch between them), then the same chain captured as a CUDA graph and replayed. Each layer is
compared with the oracle fed the GPU's previous-layer output, and the replays must reproduce
the eager outputs bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import nvfp4_mixture_experts_bf16_gb300 as moe
from _gpu_fixtures import (GAMMA_NARROW, GAMMA_WIDE, compare_outputs, dev_bf16, gamma, host_u16,
                           pack_from_experts, small_layer)
from test_gpu_parity import ALL, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.lib()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("T,H,E,k,I", [
    (1, 1152, 40, 4, 128),    # H % 256 != 0: the one-launch kernel's warps need whole k-steps
    (3, 1152, 40, 4, 128),
    (8, 1152, 40, 4, 128),
    (8, 8192, 24, 3, 64),     # the activation operand of 8 tokens does not fit beside a stage
])
def test_forward_narrow_multi_kernel_path(T, H, E, k, I, mode):
    x, wr, ex = small_layer(T, H, E, k, I, seed=71 + T, zipf=T > 1)
    pack = pack_from_experts(ex)
    r = run_and_check(x, wr, ex, pack, k, mode)
    assert r["launches"] == 4, r["launches"]   # route, gate/up, down, combine
    pack.close()


@pytest.mark.parametrize("T,H,E,k,I", [
    (40, 1152, 24, 4, 128),   # H % 256 != 0: no 256-row weight tiles for the resident h tile
    (20, 256, 8, 2, 1536),    # the h tile of I = 1536 (192 KB in f16) does not stay resident
])
def test_forward_w4a16_wide_down_restaged(T, H, E, k, I):
    x, wr, ex = small_layer(T, H, E, k, I, seed=81 + T, zipf=True)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, 0)
    pack.close()


@pytest.mark.parametrize("T,H,E,k,I,mode", [
    (40, 1152, 24, 4, 128, 1),   # W4A4, H % 256 != 0: no tcgen05 FP4 tiles
    (30, 512, 16, 3, 192, 0),    # W4A16, I % 128 != 0: no tcgen05 f16 tiles
])
def test_forward_wide_grouped_mma_sync_path(T, H, E, k, I, mode):
    x, wr, ex = small_layer(T, H, E, k, I, seed=91 + T, zipf=True)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, mode)
    pack.close()


@pytest.mark.parametrize("T,H,E,k,I", [
    (60, 256, 4, 2, 64),      # h resident: 1 K chunk and 1 scale-factor atom; one gate/up tile
    (300, 512, 6, 2, 320),    # h resident: 5 scale-factor atoms, 2 K chunks
    (200, 256, 4, 2, 512),    # h resident: 8 scale-factor atoms
    (150, 256, 4, 2, 768),    # two h tiles do not fit beside two weight tiles: h restaged per unit
])
def test_forward_w4a4_wide_down_variants(T, H, E, k, I):
    # the W4A4 down GEMM keeps a token tile's h in shared memory while its CTA runs the expert's
    # weight tiles, over ranges of units that straddle token tiles; large I restages h instead
    x, wr, ex = small_layer(T, H, E, k, I, seed=97 + I, zipf=True)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, 1)
    pack.close()


@pytest.mark.parametrize("mode", [0, 2])
@pytest.mark.parametrize("T,H,E,k,I", [
    (45, 256, 3, 2, 128),     # one token tile per expert, 30 slots: 16-row box + 14 plain rows
    (300, 512, 6, 2, 384),    # ~100 slots per expert (Zipf): 32-row boxes and ragged tails
    (200, 256, 4, 2, 512),    # h tile of 128 KB: no room for the Y staging, plain row stores
])
def test_forward_w4a16_wide_down_y_stores(T, H, E, k, I, mode):
    x, wr, ex = small_layer(T, H, E, k, I, seed=131 + I + mode, zipf=True)
    pack = pack_from_experts(ex)
    run_and_check(x, wr, ex, pack, k, mode)
    pack.close()


@pytest.mark.parametrize("T,H,I", [(3, 1152, 128), (40, 512, 192)])
def test_forward_w4a8_outside_its_paths_is_unsupported(T, H, I):
    # W4A8 runs on the fused narrow kernel and the tensor-core f16 path; the narrow multi-kernel
    # path (H % 256 != 0) and the grouped mma.sync path (I % 128 != 0) refuse it
    x, wr, ex = small_layer(T, H, 16, 2, I, seed=96)
    pack = pack_from_experts(ex)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, 2, 2)
    assert e.value.code == 2     # MOE_ERR_UNSUPPORTED
    pack.close()


def test_forward_w4a4_unequal_input_scales_is_unsupported():
    T, H, E, k, I = 4, 256, 8, 2, 64
    x, wr, ex = small_layer(T, H, E, k, I, seed=95)
    ex.in_scale[3, 1] *= 2.0     # one up matrix with its own input scale
    pack = pack_from_experts(ex)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, k, 1)
    assert e.value.code == 2     # MOE_ERR_UNSUPPORTED
    out = moe.moe_forward(dev_bf16(x), dev_bf16(wr), pack, k, 0)   # W4A16 ignores input scales
    torch.cuda.synchronize()
    ref = oracle.forward(x, wr, ex, k, 0)
    compare_outputs(host_u16(out), ref, 0, range(T))
    pack.close()


def _chain(layers, x0, T, k, mode):
    """Runs the layers chained (out_l is x_{l+1}) on one stream and workspace; returns the
    [L+1, T, H] activations tensor, the step function, the stream and the workspace."""
    L, H = len(layers), x0.shape[1]
    wrs = [dev_bf16(wr) for wr, _, _ in layers]
    xs = torch.empty((L + 1, T, H), dtype=torch.bfloat16, device="cuda")
    xs[0] = dev_bf16(x0)
    ws = moe.new_workspace(max(moe.moe_workspace_size(p, T, k, mode) for _, _, p in layers))
    s = torch.cuda.Stream()

    def chain():
        for l, (_, _, pack) in enumerate(layers):
            moe.moe_forward(xs[l], wrs[l], pack, k, mode, out=xs[l + 1], ws=ws, stream=s)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    return xs, chain, s, ws


@pytest.mark.parametrize("T,mode", [(1, 0), (5, 1), (40, 1), (40, 0)])
def test_chained_layers_eager_and_graph(T, mode):
    L, H, E, k, I = 4, 512, 64, 4, 128
    layers = []
    for l in range(L):
        x, wr, ex = small_layer(T, H, E, k, I, seed=100 + l, zipf=T > 1)
        layers.append((wr, ex, pack_from_experts(ex)))
    x0 = small_layer(T, H, E, k, I, seed=100, zipf=T > 1)[0]
    if mode == 1:
        # W4A4 input scales are calibrations of the activations a matrix sees; a layer's output
        # is far smaller than the N(0,1) inputs the synthetic scales assume, so each layer is
        # calibrated on its own input in a W4A16 run of the chain: the x scale from that input's
        # amax, the down scale from the amax of h over the slots it routes
        xs16, _, _, _ = _chain(layers, x0, T, k, 0)
        cal = host_u16(xs16)
        for l, (wr, ex, pack) in enumerate(layers):
            pack.close()
            r = oracle.forward(cal[l], wr, ex, k, 0, nthreads=8, want=("h",))
            xs_l = float(np.float32(np.abs(synth.bf16_to_f32(cal[l])).max()) / np.float32(2688))
            hs_l = float(np.float32(np.abs(r["h"]).max()) / np.float32(2688))
            ex.in_scale[:, 0] = xs_l
            ex.in_scale[:, 1] = xs_l
            ex.in_scale[:, 2] = hs_l
            layers[l] = (wr, ex, pack_from_experts(ex))
    xs, chain, s, ws = _chain(layers, x0, T, k, mode)
    assert moe.moe_read_device_status(ws) == 0
    eager = host_u16(xs)
    for l, (wr, ex, _) in enumerate(layers):
        ref = oracle.forward(eager[l], wr, ex, k, mode, nthreads=8, want=ALL)
        # tokens whose k-th and (k+1)-th oracle logits lie within the router's FP32 error bound
        # may select either expert: not compared. W4A4: the intermediate h codes of a chained
        # layer are not read back, so every flagged h decision may have flipped: each token's
        # bound widens by the oracle's flip allowances of all its slots (triangle inequality).
        toks, allow = [], {}
        gm = gamma(GAMMA_NARROW if T <= 8 else GAMMA_WIDE)
        for t in range(T):
            order = np.argsort(-ref["logits"][t], kind="stable")
            a, b = order[k - 1], order[k]
            if ref["logits"][t, a] - ref["logits"][t, b] <= \
                    gm * (ref["abssum"][t, a] + ref["abssum"][t, b]):
                continue
            toks.append(t)
            if mode == 1:
                a = 0.0
                for j in range(k):
                    sl = ref["slot_of"][t, j]
                    a += ref["w"][t, j] * (ref["h_amb_elem"][sl].sum() + ref["h_amb_block"][sl].sum())
                allow[t] = a
        assert len(toks) >= max(1, T - 2), (l, len(toks))
        assert np.abs(synth.bf16_to_f32(eager[l + 1])).max() > 0   # the chain carries signal
        compare_outputs(eager[l + 1], ref, mode, toks, allow)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for _ in range(2):
        xs[1:].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(xs), eager)
    assert moe.moe_read_device_status(ws) == 0
    for _, _, p in layers:
        p.close()
