"""GPU parity of moe_forward_layers: a stack of layers chained in one call through the residual
stream (layer l+1's input is BF16(layer l's input + its output)), one launch of the fused kernel
per layer on narrow calls (its combine writing the residual sum). Its outputs must equal, bit for
bit, those of one moe_forward call per layer fed the same residual sums (each of which the main
parity tests compare with the oracle), and each layer is also compared with the oracle directly.
A long stack, shapes outside the fused kernel (one launch sequence per layer plus the residual
sum), CUDA-graph replay and the full-size decode shapes are covered too."""
import numpy as np
import pytest
import torch

import oracle
import synth
import nvfp4_mixture_experts_bf16_gb300 as moe
from _gpu_fixtures import (GAMMA_NARROW, GAMMA_WIDE, FullLayer, compare_outputs, dev_bf16,
                           gamma, host_u16, pack_from_experts, small_layer, ws_array)
from test_gpu_parity import ALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    moe.lib()


def _stack(L, T, H, E, k, I, mode, seed):
    """L layers (router, oracle experts, pack) and the first layer's input."""
    layers = []
    for l in range(L):
        _, wr, ex = small_layer(T, H, E, k, I, seed=seed + l, zipf=T > 1)
        layers.append([wr, ex, pack_from_experts(ex)])
    x0 = small_layer(T, H, E, k, I, seed=seed, zipf=T > 1)[0]
    return layers, x0


def residual(x, out):
    """BF16(x + out) of two BF16 tensors: the FP32 sum rounded to nearest even."""
    return (x.float() + out.float()).to(torch.bfloat16)


def _sequential(layers, x0, k, mode):
    """One moe_forward call per layer, fed the residual sums: (inputs [L, T, H], outputs
    [L, T, H]) as host BF16 bits."""
    xs, outs = [dev_bf16(x0)], []
    for wr, _, pack in layers:
        outs.append(moe.moe_forward(xs[-1], dev_bf16(wr), pack, k, mode))
        xs.append(residual(xs[-1], outs[-1]))
    torch.cuda.synchronize()
    return np.stack([host_u16(t) for t in xs[:-1]]), np.stack([host_u16(t) for t in outs])


def _check_oracle(layers, xs, outs, k, mode):
    """Each layer's output against the oracle fed that layer's GPU input (near ties of the router
    and W4A4 h flips handled as in the chained-layer test of test_gpu_branches)."""
    T = xs.shape[1]
    gm = gamma(GAMMA_NARROW if T <= 8 else GAMMA_WIDE)
    for l, (wr, ex, _) in enumerate(layers):
        ref = oracle.forward(xs[l], wr, ex, k, mode, nthreads=8, want=ALL)
        toks, allow = [], {}
        for t in range(T):
            order = np.argsort(-ref["logits"][t], kind="stable")
            a, b = order[k - 1], order[k]
            if ref["logits"][t, a] - ref["logits"][t, b] <= gm * (ref["abssum"][t, a] +
                                                                  ref["abssum"][t, b]):
                continue
            toks.append(t)
            if mode in (1, 2):   # W4A4 element and block flips; W4A8 element flips
                allow[t] = sum(ref["w"][t, j] * (ref["h_amb_elem"][ref["slot_of"][t, j]].sum() +
                                                 ref["h_amb_block"][ref["slot_of"][t, j]].sum())
                               for j in range(k))
        assert len(toks) >= max(1, T - 2), (l, len(toks))
        assert np.abs(synth.bf16_to_f32(outs[l])).max() > 0
        compare_outputs(outs[l], ref, mode, toks, allow)


@pytest.mark.parametrize("T,mode", [(1, 0), (1, 1), (2, 0), (5, 1), (8, 0), (1, 2), (6, 2)])
def test_layers_fused_equal_single_calls_and_oracle(T, mode):
    L, H, E, k, I = 5, 512, 64, 4, 128
    layers, x0 = _stack(L, T, H, E, k, I, mode, seed=200 + T)
    xs, seq = _sequential(layers, x0, k, mode)
    packs = [p for _, _, p in layers]
    ws = moe.new_workspace(moe.moe_workspace_size_layers(packs[0], L, T, k, mode))
    out = moe.moe_forward_layers(dev_bf16(x0), [dev_bf16(wr) for wr, _, _ in layers], packs, k,
                                 mode, ws=ws)
    assert moe.moe_last_launch_count() == L      # one launch of the fused kernel per layer
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    got = host_u16(out)
    assert np.array_equal(got, seq)
    _check_oracle(layers, xs, got, k, mode)
    # each layer's routing sits in its own workspace region: the oracle's selection
    for l, (wr, ex, _) in enumerate(layers):
        off = moe.moe_workspace_offsets_layers(packs[0], L, T, k, mode, l)
        idx = ws_array(ws, off["idx"], T * k * 4, np.int32).reshape(T, k)
        ref = oracle.route(xs[l], wr, k)
        same = [t for t in range(T) if np.array_equal(idx[t], ref["idx"][t])]
        assert len(same) >= max(1, T - 2)
    for p in packs:
        p.close()


def test_layers_long_stack():
    # 40 chained layers
    L, T, H, E, k, I = 40, 2, 256, 16, 2, 64
    layers, x0 = _stack(L, T, H, E, k, I, 0, seed=300)
    _, seq = _sequential(layers, x0, k, 0)
    packs = [p for _, _, p in layers]
    out = moe.moe_forward_layers(dev_bf16(x0), [dev_bf16(wr) for wr, _, _ in layers], packs, k, 0)
    assert moe.moe_last_launch_count() == L
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), seq)
    for p in packs:
        p.close()


@pytest.mark.parametrize("T,mode", [(3, 0), (3, 1), (20, 1), (20, 0)])
def test_layers_outside_the_fused_kernel(T, mode):
    # H % 256 != 0 (narrow) and wide calls: one launch sequence per layer, same results
    L, H, E, k, I = 3, 1152 if T <= 8 else 512, 32, 3, 128
    layers, x0 = _stack(L, T, H, E, k, I, mode, seed=400 + T)
    _, seq = _sequential(layers, x0, k, mode)
    packs = [p for _, _, p in layers]
    out = moe.moe_forward_layers(dev_bf16(x0), [dev_bf16(wr) for wr, _, _ in layers], packs, k,
                                 mode)
    assert moe.moe_last_launch_count() > L
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), seq)
    for p in packs:
        p.close()


def test_layers_graph_replay_and_repeat():
    L, T, H, E, k, I = 6, 1, 512, 64, 4, 128
    layers, x0 = _stack(L, T, H, E, k, I, 0, seed=500)
    _, seq = _sequential(layers, x0, k, 0)
    packs = [p for _, _, p in layers]
    wrs = [dev_bf16(wr) for wr, _, _ in layers]
    x = dev_bf16(x0)
    out = torch.empty((L, T, H), dtype=torch.bfloat16, device="cuda")
    ws = moe.new_workspace(moe.moe_workspace_size_layers(packs[0], L, T, k, 0))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):      # the workspace is reused call after call without re-zeroing
            moe.moe_forward_layers(x, wrs, packs, k, 0, out=out, ws=ws, stream=s)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), seq)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_forward_layers(x, wrs, packs, k, 0, out=out, ws=ws, stream=s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_u16(out), seq)
    assert moe.moe_read_device_status(ws) == 0
    for p in packs:
        p.close()


def test_layers_rejects_bad_arguments():
    L, T, H, E, k, I = 2, 1, 256, 16, 2, 64
    layers, x0 = _stack(L, T, H, E, k, I, 0, seed=600)
    packs = [p for _, _, p in layers]
    wrs = [dev_bf16(wr) for wr, _, _ in layers]
    x = dev_bf16(x0)
    _, _, ex = small_layer(T, 512, E, k, I, seed=601)
    other = pack_from_experts(ex)                       # a pack of another hidden size
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_layers(x, wrs, [packs[0], other], k, 0)
    assert e.value.code == 1
    out = torch.empty((L, T, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:              # x inside the outputs
        moe.moe_forward_layers(out[1], wrs, packs, k, 0, out=out)
    assert e.value.code == 1
    small = moe.new_workspace(moe.moe_workspace_size_layers(packs[0], 1, T, k, 0))
    with pytest.raises(moe.MoeError) as e:              # a workspace for one layer only
        moe.moe_forward_layers(x, wrs, packs, k, 0, ws=small)
    assert e.value.code == 6
    other.close()
    for p in packs:
        p.close()


def test_layers_full_size_decode():
    # the decode shapes (H 4096, 512 experts, top-10, I 384): three chained layers
    L, T, k = 3, 1, 10
    lays = [FullLayer(0, l, T, False) for l in range(L)]
    x0 = lays[0].x
    xs, outs = [dev_bf16(x0)], []
    for lay in lays:
        outs.append(moe.moe_forward(xs[-1], dev_bf16(lay.wr), lay.pack, k, 0))
        xs.append(residual(xs[-1], outs[-1]))
    torch.cuda.synchronize()
    seq = np.stack([host_u16(t) for t in outs])
    xin = np.stack([host_u16(t) for t in xs[:-1]])
    out = moe.moe_forward_layers(dev_bf16(x0), [dev_bf16(lay.wr) for lay in lays],
                                 [lay.pack for lay in lays], k, 0)
    assert moe.moe_last_launch_count() == L
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), seq)
    # each layer against the oracle (its selected experts, quantised by the oracle)
    for l, lay in enumerate(lays):
        r = oracle.route(xin[l], lay.wr, k)
        ex = lay.oracle_experts(r["idx"].ravel())
        ref = oracle.forward(xin[l], lay.wr, ex, k, 0, nthreads=8,
                             want=("out_bf16", "logits", "abssum", "idx", "w"))
        order = np.argsort(-ref["logits"][0], kind="stable")
        a, b = order[k - 1], order[k]
        if ref["logits"][0, a] - ref["logits"][0, b] > \
                gamma(GAMMA_NARROW) * (ref["abssum"][0, a] + ref["abssum"][0, b]):
            compare_outputs(seq[l], ref, 0, range(T))
        lay.close()
