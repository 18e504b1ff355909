#!/usr/bin/env python3
"""Benchmark of the GB300 NVFP4 routed-expert MoE step (one JSON line on stdout).

Headline workload (``decode1``): one decode step of a 48-layer stack, 1 token per layer, W4A16,
hidden 4096, 512 experts, top-10, expert intermediate 384; every layer has its own router and its
own 512-expert NVFP4 pack (65 GB resident), so a step streams 48 x 10 selected experts
(1.27 GB) and nothing is reused from L2 between steps. A "step" = the 48 layers, captured in
one CUDA graph (PDL-chained kernels). ``value`` = layer-tokens per second = T * layers / step
time. Inputs are seeded synthetic (``synth``), resident in HBM before timing starts.

Also reported in the same line: the roofline of the dominant kernel from CUDA events on its
stream (for narrow calls the whole step is one persistent kernel, ``k_decode``, so its mean
launch time is the timed step / layers), the end-to-end number through the C ABI with host buffers
(host->device copy of x and device->host copy of out inside the timed region), the SM clocks
sampled during the timed region, a secondary table (8-token verify W4A16/W4A4 and the
8192-token prefill), and the CPU oracle timed on a bounded sample as a reported baseline.

``--impl reference`` times the CPU oracle alone (the reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer tokens/s + HBM GB/s (decode), NVFP4 TFLOPS (prefill), % roofline"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--workload", default="decode1", choices=list(synth.WORKLOADS))
    p.add_argument("--layers", type=int, default=None)
    p.add_argument("--tokens", type=int, default=None, help="tokens per layer (profiling)")
    p.add_argument("--experts", type=int, default=None,
                   help="experts per layer (smaller packs for profiler captures)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--mode", default=None, choices=["w4a16", "w4a4", "w4a8"],
                   help="override the workload's activation mode (profiling)")
    p.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--shared", action="store_true",
                   help="time the step with a BF16 shared expert per layer (Is = I)")
    return p.parse_args()


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=smax,
                    reasons=sorted(reasons), samples=len(sm))


# Sources each profiled kernel is compiled from; a committed DRAM count is quoted only while
# these files are byte-identical to the ones the capture ran.
KERNEL_SOURCES = {
    "k_decode": ("moe_decode.cu", "moe_internal.cuh"),
    "k_gateup": ("moe_experts.cu", "moe_internal.cuh"),
}


def source_sha(kernel=None):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_mixture_experts_bf16_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(csrc))
    for n in names:
        h.update(open(os.path.join(csrc, n), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(f"{kernel}:{workload}")
    if not d or d.get("source_sha") != source_sha(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def bytes_gateup(U, H, I):
    return U * (2 * I * H // 2 + 2 * I * H // 16)


def bytes_down(U, H, I):
    return U * (H * I // 2 + H * I // 16)


def bytes_decode_launch(U, T, H, E, I):
    """Algorithmic DRAM bytes of one fused narrow-call launch: the router (read once), every
    selected expert's NVFP4 codes + scales + 3 multipliers (each read once), x in and out out."""
    return E * H * 2 + bytes_gateup(U, H, I) + bytes_down(U, H, I) + U * 12 + 2 * T * H * 2


# ------------------------------------------------------------------ CPU oracle (baseline arm)
def oracle_sample(wl, seed, n_tokens, threads):
    """A bounded sample of the workload for the CPU oracle: n_tokens tokens of layer 0 with the
    experts they select (generated and quantised outside the timed region)."""
    import oracle
    H, E, k, I = wl.H, wl.E, wl.k, wl.I
    x = synth.activations(seed, 0, n_tokens, H, wl.zipf)
    wr = synth.router_weight(seed, 0, E, H, wl.zipf)
    r = oracle.route(x, wr, k, nthreads=threads)
    ex = oracle.ExpertSet(E, H, I)
    xs = synth.activation_input_scale(H)
    ds = synth.down_input_scales(seed, 0, E)
    for e in sorted(set(r["idx"].ravel().tolist())):
        q = [oracle.quantize_weight_bf16(synth.expert_weight(seed, 0, e, w, H, I), nthreads=threads)
             for w in ("gate", "up", "down")]
        ex.set(e, q[0][:2], q[1][:2], q[2][:2], (q[0][2], q[1][2], q[2][2]), (xs, xs, float(ds[e])))
    return x, wr, ex


def time_oracle(wl, seed, steps, budget_s, threads, n_tokens, warmup=1):
    import oracle
    x, wr, ex = oracle_sample(wl, seed, n_tokens, threads)
    for _ in range(warmup):   # untimed: thread pool start-up and first-touch of the sample
        oracle.forward(x, wr, ex, wl.k, wl.mode, nthreads=threads, want=("out_bf16",))
    times = []
    t_end = time.time() + budget_s
    for _ in range(max(1, steps)):
        t0 = time.perf_counter()
        oracle.forward(x, wr, ex, wl.k, wl.mode, nthreads=threads, want=("out_bf16",))
        times.append(time.perf_counter() - t0)
        if time.time() > t_end:
            break
    t = statistics.median(times)
    return dict(value=n_tokens / t, unit="layer-tokens/s", cores=threads, kind="oracle",
                sample=f"{n_tokens} tokens of layer 0 of '{wl.name}' (T={wl.T} workload shapes), "
                       f"{len(times)} timed calls, median", calls=len(times))


def run_reference(args, rank, world):
    wl = synth.WORKLOADS[args.workload]
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    n_tok = 4 if wl.T <= 8 else 8
    cb = time_oracle(wl, args.seed, args.steps, budget_s=120, threads=threads, n_tokens=n_tok,
                     warmup=args.warmup)
    line = dict(impl="reference", metric=METRIC, value=cb["value"], unit=cb["unit"],
                n_gpus=world, steps=cb["calls"], warmup=args.warmup,
                ms_per_step=1e3 * n_tok / cb["value"],
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=bench_config(wl, args.layers or wl.layers, world, args),
                cpu_baseline=cb,
                e2e=dict(value=cb["value"], unit=cb["unit"], h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ multi-rank aggregation
def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's step time (every rank gets it): replicas finish when the last does."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, ms: float) -> float:
    """Whole-job layer-tokens/s: every rank processes tokens_per_step per step (weak scaling)."""
    return world * tokens_per_step / (ms / 1e3)


# ------------------------------------------------------------------ native arm
class Layer:
    def __init__(self, x, wr, pack, U, shared=None, xall=None):
        self.x, self.wr, self.pack, self.U = x, wr, pack, U
        self.shared = shared   # (gate_up, down, gate) BF16 tensors of the shared expert, or None
        self.xall = xall       # [layers, T, H]: every layer's x, of which self.x is one row


def quantized_experts(seed, layer, E, H, I, device):
    """Synthetic checkpoint of one layer drawn on the device and quantised with the library's
    own NVFP4 quantiser (multiplier = global amax / 2688 per matrix)."""
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    mats = {}
    for w in ("gate", "up", "down"):
        W = synth.torch_expert_weights(seed, layer, w, E, H, I, device)
        # multiplier = fl32(amax / 2688) by an IEEE float32 division on the host
        S = W.float().abs().amax(dim=(1, 2)).cpu().numpy().astype(np.float32) / np.float32(2688.0)
        rows, cols = W.shape[1], W.shape[2]
        codes = torch.empty((E, rows, cols // 2), dtype=torch.uint8, device=device)
        scales = torch.empty((E, rows, cols // 16), dtype=torch.uint8, device=device)
        for e in range(E):
            moe.moe_quantize_act_nvfp4(W[e], float(S[e]), codes[e], scales[e])
        del W
        mats[w] = (codes, scales, S)
    return mats


def dev_bf16(u16, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).to(device).view(torch.bfloat16)


def with_shared(stack, wl, seed, device):
    """The same layers, each with its own BF16 shared expert of intermediate size I."""
    return [Layer(L.x, L.wr, L.pack, L.U,
                  synth.torch_shared_expert_weights(seed, l, wl.H, wl.I, device), L.xall)
            for l, L in enumerate(stack)]


def bytes_shared(H, Is):
    """BF16 bytes of one shared expert: gate/up, down and the gate vector."""
    return 2 * (2 * Is * H + H * Is + H)


def build_stack(wl, layers, seed, device, packs=None):
    """layers x (x, router, pack); packs may be reused from another workload of equal shapes."""
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    out = []
    xs = synth.activation_input_scale(wl.H)
    for l in range(layers):
        x = dev_bf16(synth.activations(seed, l, wl.T, wl.H, wl.zipf), device)
        wr = dev_bf16(synth.router_weight(seed, l, wl.E, wl.H, wl.zipf), device)
        if packs is None:
            m = quantized_experts(seed, l, wl.E, wl.H, wl.I, device)
            ds = synth.down_input_scales(seed, l, wl.E)
            args = []
            for w in ("gate", "up", "down"):
                codes, scales, S = m[w]
                ins = [xs] * wl.E if w != "down" else [float(v) for v in ds]
                args.append([(codes[e], scales[e], float(S[e]), ins[e]) for e in range(wl.E)])
            pack = moe.moe_pack_nvfp4(args[0], args[1], args[2], wl.H, wl.I)
            del m, args
            torch.cuda.synchronize()
        else:
            pack = packs[l % len(packs)]
        r = moe.moe_route_topk(x, wr, wl.k)
        U = int((r["counts"] > 0).sum().item())
        out.append(Layer(x, wr, pack, U))
    # every layer's activations in one [layers, T, H] tensor (each layer's x a row of it), so a
    # step's inputs move host->device in one copy
    xall = torch.stack([L.x for L in out])
    for l, L in enumerate(out):
        L.x, L.xall = xall[l], xall
    return out


def measure(wl, stack, steps, warmup, use_graph, device, clocks=None):
    """Time `steps` steps (all layers) on one stream; returns per-step ms and the launch count."""
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    s = torch.cuda.Stream(device=device)
    sh = stack[0].shared
    nws = (moe.moe_workspace_size(stack[0].pack, wl.T, wl.k, wl.mode) if sh is None else
           moe.moe_workspace_size_shared(stack[0].pack, wl.T, wl.k, wl.mode, sh[0].shape[0] // 2))
    ws = moe.new_workspace(nws, device)
    oall = torch.empty((len(stack), wl.T, wl.H), dtype=torch.bfloat16, device=device)
    outs = list(oall)           # each layer's out is a row of one tensor (one device->host copy)
    launches = [0]

    def step():
        n = 0
        for L, o in zip(stack, outs):
            if L.shared is None:
                moe.moe_forward(L.x, L.wr, L.pack, wl.k, wl.mode, out=o, ws=ws, stream=s)
            else:
                moe.moe_forward_shared(L.x, L.wr, L.pack, L.shared, wl.k, wl.mode, out=o, ws=ws,
                                       stream=s)
            n += moe.moe_last_launch_count()
        launches[0] = n

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step
    with torch.cuda.stream(s):
        for _ in range(warmup):
            run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.start()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):
            run()
        e1.record(s)
    torch.cuda.synchronize()
    info = clocks.stop() if clocks else None
    status = moe.moe_read_device_status(ws, stream=s)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    return e0.elapsed_time(e1) / steps, launches[0], info, (s, ws, oall, run, step)


def measure_stack(wl, stack, steps, warmup, use_graph, device, clocks=None):
    """Time `steps` steps of the layers chained through the residual stream with
    moe_forward_layers (layer 0 reads stack[0].x; layer l+1 reads BF16(x_l + out_l)); returns
    per-step ms, launches per step, the clock record, the mean distinct experts per layer (from
    each layer's counts in the workspace) and the state for the end-to-end measurement."""
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    s = torch.cuda.Stream(device=device)
    L = len(stack)
    packs = [Lr.pack for Lr in stack]
    wrs = [Lr.wr for Lr in stack]
    x = stack[0].x.clone()
    out = torch.empty((L, wl.T, wl.H), dtype=torch.bfloat16, device=device)
    ws = moe.new_workspace(moe.moe_workspace_size_layers(packs[0], L, wl.T, wl.k, wl.mode), device)
    launches = [0]

    def step():
        moe.moe_forward_layers(x, wrs, packs, wl.k, wl.mode, out=out, ws=ws, stream=s)
        launches[0] = moe.moe_last_launch_count()

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    U = []
    for l in range(L):
        off = moe.moe_workspace_offsets_layers(packs[0], L, wl.T, wl.k, wl.mode, l)
        c = ws[off["counts"]:off["counts"] + 4 * wl.E].cpu().numpy().view(np.int32)
        U.append(int((c > 0).sum()))
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step
    with torch.cuda.stream(s):
        for _ in range(warmup):
            run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.start()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):
            run()
        e1.record(s)
    torch.cuda.synchronize()
    info = clocks.stop() if clocks else None
    if moe.moe_read_device_status(ws, stream=s) != 0:
        raise RuntimeError("device status after the timed region")
    return e0.elapsed_time(e1) / steps, launches[0], info, float(np.mean(U)), \
        (s, x, out, run, step)


def e2e_stack(wl, L, steps, state, use_graph=True):
    """The chained stack end to end: per step the first layer's input host->device, the step,
    every layer's output device->host (pinned buffers)."""
    import torch
    s, x, out, run, step = state
    if not use_graph:
        run = step
    hx = x.cpu().pin_memory()
    ho = torch.empty(tuple(out.shape), dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for it in range(steps + 2):
            if it == 2:
                e0.record(s)
            x.copy_(hx, non_blocking=True)
            run()
            ho.copy_(out, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, wl.T * wl.H * 2, L * wl.T * wl.H * 2


def kernel_label(name):
    """A short label of a kernel name as cudaFuncGetName returns it (mangled or not)."""
    import re
    if not name:
        return "?"
    m = re.search(r"(k_[A-Za-z0-9_]+?)(I(?:L[a-z](-?\d+)E)+E)?(?:E|v|$)", name)
    if m is None:
        m2 = re.search(r"(k_[A-Za-z0-9_]+)(<[^>]*>)?", name)
        return m2.group(0) if m2 else name[:40]
    args = re.findall(r"L[a-z](-?\d+)E", m.group(2) or "")
    return m.group(1) + (f"<{','.join(args)}>" if args else "")


def launch_times(wl, stack, reps, device):
    """Mean device time of each kernel launch of one forward call (per layer), from CUDA events
    recorded around every launch on the launching stream (programmatic dependent launch off
    while profiling): [(kernel, ms)]."""
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    s = torch.cuda.Stream(device=device)
    sh = stack[0].shared
    nws = (moe.moe_workspace_size(stack[0].pack, wl.T, wl.k, wl.mode) if sh is None else
           moe.moe_workspace_size_shared(stack[0].pack, wl.T, wl.k, wl.mode, sh[0].shape[0] // 2))
    ws = moe.new_workspace(nws, device)
    outs = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device) for _ in stack]
    acc, names, n = None, None, 0
    with torch.cuda.stream(s):
        for rep in range(reps + 1):
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(64)] for _ in stack]
            for ev in evs:          # torch creates the CUDA event at its first record
                for e in ev:
                    e.record(s)
            nl = []
            for L, o, ev in zip(stack, outs, evs):
                moe.moe_profile_next_forward(ev)
                if L.shared is None:
                    moe.moe_forward(L.x, L.wr, L.pack, wl.k, wl.mode, out=o, ws=ws, stream=s)
                else:
                    moe.moe_forward_shared(L.x, L.wr, L.pack, L.shared, wl.k, wl.mode, out=o,
                                           ws=ws, stream=s)
                nl.append(min(moe.moe_last_launch_count(), 32))
            names = [kernel_label(moe.moe_profile_kernel_name(i)) for i in range(nl[-1])]
            torch.cuda.synchronize()
            if rep == 0:
                continue  # warm-up
            for ev, k in zip(evs, nl):
                t = np.array([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(k)])
                acc = t if acc is None else acc + t
                n += 1
    return list(zip(names, (acc / n).tolist()))


def e2e_measure(wl, stack, steps, state, device, use_graph=True):
    """Same metric through the public API with host buffers: per step, copy every layer's x
    host->device (pinned; the layers' inputs are one [layers, T, H] buffer, so one copy), run
    the step (the captured graph, or with use_graph=False every moe_forward call issued from
    the host as a caller without graphs would), copy every layer's out device->host (one copy of
    the [layers, T, H] outputs)."""
    import torch
    s, ws, oall, run, step = state
    if not use_graph:
        run = step
    xall = stack[0].xall
    assert all(L.xall is xall for L in stack)
    hx = xall.cpu().pin_memory()
    ho = torch.empty(tuple(oall.shape), dtype=torch.bfloat16).pin_memory()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for it in range(steps + 2):
            if it == 2:
                e0.record(s)
            xall.copy_(hx, non_blocking=True)
            run()
            ho.copy_(oall, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    nbytes = len(stack) * wl.T * wl.H * 2
    return ms, nbytes


def bench_config(wl, layers, world, args):
    """The workload description both arms print (the same dict, so the lines compare)."""
    return dict(workload=wl.name, T=wl.T, layers=layers, hidden=wl.H, experts=wl.E, top_k=wl.k,
                inter=wl.I, mode=["W4A16", "W4A4", "W4A8"][wl.mode],
                parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                l2=("no flush: a step streams 48 layers x 10 experts = 1.27 GB > 129 MB L2"
                    if wl.T == 1 and layers >= 48 else
                    "no flush: a step streams more expert bytes than the 129 MB L2 holds"),
                graph=not args.no_graph, shared_expert=bool(args.shared))


# FP4 dense tensor peak from the measured BF16 peak and NVIDIA's nominal dense ratio for GB300
# (FP4 13.5 PFLOP/s : BF16 2.25 PFLOP/s = 6)
FP4_PER_BF16 = 6.0


def prefill_roofline(w3, ms3, kernels, U, pk, shared):
    """The prefill chunk against both of its roofs: the tensor peak of its MMA kind (FP4 for
    W4A4, BF16/FP16 for W4A16) and HBM for the bytes it must move at least once (the touched
    experts' NVFP4 weights, the router, x in and out out); plus the dominant kernel (live per-
    launch CUDA events) with its own FLOPs against the same peak."""
    H, I, T, E, k = w3.H, w3.I, w3.T, w3.E, w3.k
    gu_flops = 2 * T * k * 2 * I * H
    dn_flops = 2 * T * k * I * H
    flops = gu_flops + dn_flops
    if w3.mode == 1:
        peak = pk["bf16"] * FP4_PER_BF16
        src = (f"{pk['src']} bf16_tflops {pk['bf16']} x {FP4_PER_BF16:g} (nominal dense "
               "FP4:BF16 ratio, 13.5:2.25 PFLOP/s)")
    else:
        peak = pk["bf16"]
        src = f"{pk['src']} bf16_tflops (kind::f16 runs at the BF16/FP16 rate)"
    floor = U * (bytes_gateup(1, H, I) + bytes_down(1, H, I) + 12) + E * H * 2 + 2 * T * H * 2
    tot = sum(t for _, t in kernels) or 1.0
    dom_name, dom_ms = max(kernels, key=lambda kv: kv[1]) if kernels else ("?", 0.0)
    dom_flops = (gu_flops if ("<0>" in dom_name or "<false>" in dom_name) and
                 ("k_tc_gemm" in dom_name or "k_tc16" in dom_name) and "dn" not in dom_name
                 else dn_flops if ("k_tc_gemm<1>" in dom_name or "k_tc_down" in dom_name or
                                   "k_tc16_dn" in dom_name or "k_tc16<1>" in dom_name) else None)
    achieved = flops / (ms3 * 1e-3) / 1e12
    r = dict(bound="hbm" if floor / (pk["hbm"] * 1e9) > flops / (peak * 1e12) else "tensor",
             achieved=round(achieved, 1), peak=round(peak, 1), unit="TFLOP/s",
             frac=round(achieved / peak, 4), peak_source=src,
             flops_per_chunk=flops,
             hbm=dict(bytes_floor=int(floor), achieved_gbs=round(floor / (ms3 * 1e-3) / 1e9, 1),
                      peak=pk["hbm"], frac=round(floor / (ms3 * 1e-3) / 1e9 / pk["hbm"], 4),
                      floor_ms=round(floor / (pk["hbm"] * 1e9) * 1e3, 4),
                      note="touched experts' NVFP4 weights + router + x + out, each once"),
             # the chunk's time against the larger of its two floors
             bound_ms=round(max(flops / (peak * 1e12), floor / (pk["hbm"] * 1e9)) * 1e3, 4),
             frac_of_bound=round(max(flops / (peak * 1e12), floor / (pk["hbm"] * 1e9)) * 1e3 / ms3,
                                 4),
             dominant=dict(kernel=dom_name, ms=round(dom_ms, 4), share=round(dom_ms / tot, 4)),
             kernels=[dict(kernel=n, ms=round(t, 4), share=round(t / tot, 4)) for n, t in kernels],
             kernel_timing="CUDA events around each launch, PDL off (serialised)")
    if dom_flops:
        kt = dom_flops / (dom_ms * 1e-3) / 1e12
        r["dominant"].update(tflops=round(kt, 1), frac=round(kt / peak, 4))
    if shared:
        r["note"] = "achieved counts the routed FLOPs only"
    return r


def run_native(args, rank, world, local_rank):
    import torch
    import nvfp4_mixture_experts_bf16_gb300 as moe
    moe.build()
    moe.lib()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    wl = synth.WORKLOADS[args.workload]
    if args.experts or args.tokens or args.mode:
        mode = wl.mode if args.mode is None else {"w4a16": 0, "w4a4": 1, "w4a8": 2}[args.mode]
        wl = synth.Workload(wl.name, args.tokens or wl.T, wl.H, args.experts or wl.E, wl.k, wl.I,
                            mode, wl.layers, wl.zipf)
    layers = args.layers or wl.layers
    pk = peaks()
    t_setup = time.time()
    stack = build_stack(wl, layers, args.seed + 1000 * rank, device)
    if args.shared:
        stack = with_shared(stack, wl, args.seed + 1000 * rank, device)
    setup_s = time.time() - t_setup

    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local_rank) if rank == 0 else None
    ms, launches, clk, state = measure(wl, stack, args.steps, args.warmup, not args.no_graph,
                                       device, clocks)
    if world > 1:
        ms = max_over_ranks(ms, device)
    tokens_per_step = wl.T * layers
    value = job_throughput(world, tokens_per_step, ms)

    U_mean = float(np.mean([L.U for L in stack]))
    gu_bytes = bytes_gateup(U_mean, wl.H, wl.I)
    dn_bytes = bytes_down(U_mean, wl.H, wl.I)
    layer_bytes = gu_bytes + dn_bytes + (bytes_shared(wl.H, wl.I) if args.shared else 0)
    layer_s = ms / layers * 1e-3
    layer_gbs = layer_bytes / layer_s / 1e9
    peak_src = (f"{pk['src']} hbm_gbs (MEASURED_PEAKS.json)" if pk["src"] == "measured"
                else "fallback 6.8 TB/s")
    fused = launches == layers   # one launch per layer: the persistent narrow-call kernel
    kern = None
    if args.shared:
        # the whole step (shared-expert kernels + the narrow-call kernel, or the wide path)
        gbs = layer_bytes / layer_s / 1e9
        roofline = dict(bound="hbm", kernel=f"whole step with the shared expert "
                        f"({launches // layers} launches per layer)",
                        achieved=round(gbs, 1), peak=pk["hbm"], unit="GB/s",
                        frac=round(gbs / pk["hbm"], 4), traffic=None,
                        algorithmic_bytes_per_launch=None,
                        algorithmic_bytes_per_layer=int(layer_bytes), peak_source=peak_src)
    elif fused:
        # the only kernel of the step: mean launch duration = event-timed step / launches.
        # achieved = the selected experts' bytes (U x B_e, each read once), the router and the
        # activations beside it
        exp_bytes = gu_bytes + dn_bytes + 12 * U_mean
        dec_bytes = bytes_decode_launch(U_mean, wl.T, wl.H, wl.E, wl.I)
        gbs = exp_bytes / layer_s / 1e9
        gbs_r = dec_bytes / layer_s / 1e9
        roofline = dict(bound="hbm", kernel="k_decode (whole narrow-call step, one launch)",
                        achieved=round(gbs, 1), peak=pk["hbm"], unit="GB/s",
                        frac=round(gbs / pk["hbm"], 4),
                        traffic=committed_traffic("k_decode", wl.name),
                        algorithmic_bytes_per_launch=int(exp_bytes),
                        bytes_counted="selected experts' NVFP4 codes, scales and multipliers",
                        achieved_incl_router=round(gbs_r, 1),
                        frac_incl_router=round(gbs_r / pk["hbm"], 4),
                        bytes_incl_router=int(dec_bytes),
                        launch_us=round(layer_s * 1e6, 3), peak_source=peak_src)
    else:
        kern = launch_times(wl, stack, reps=3, device=device)
        dom, dom_ms = max(kern, key=lambda kv: kv[1])
        tot = sum(t for _, t in kern)
        is_gu = "gateup" in dom or (("<0>" in dom or "<false>" in dom) and "k_tc" in dom)
        is_dn = "down" in dom or "_dn" in dom or "k_tc_gemm<1>" in dom or "k_tc16<1>" in dom
        b = gu_bytes if is_gu else (dn_bytes if is_dn else gu_bytes + dn_bytes)
        kgbs = b / (dom_ms * 1e-3) / 1e9
        roofline = dict(bound="hbm", kernel=dom, achieved=round(kgbs, 1), peak=pk["hbm"],
                        unit="GB/s", frac=round(kgbs / pk["hbm"], 4),
                        traffic=committed_traffic(dom.split("<")[0], wl.name),
                        algorithmic_bytes_per_launch=int(b), launch_us=round(dom_ms * 1e3, 3),
                        share=round(dom_ms / tot, 4), peak_source=peak_src)
    e2e_ms, io_bytes = e2e_measure(wl, stack, max(3, args.steps // 2), state, device)
    e2e_ng_ms, _ = e2e_measure(wl, stack, max(3, args.steps // 2), state, device,
                               use_graph=False)

    extra = {}
    if not args.no_extra and not args.shared and rank == 0:
        packs = [L.pack for L in stack]
        for name in ("verify8", "verify8_w4a4", "verify8_w4a8"):
            w2 = synth.WORKLOADS[name]
            st2 = build_stack(w2, layers, args.seed, device, packs=packs)
            ms2, _, _, _ = measure(w2, st2, max(3, args.steps // 2), 3, not args.no_graph, device)
            U2 = float(np.mean([L.U for L in st2]))
            b2 = bytes_gateup(U2, w2.H, w2.I) + bytes_down(U2, w2.H, w2.I)
            extra[name] = dict(tokens_per_s=round(w2.T * layers / (ms2 / 1e3), 1),
                               us_per_layer=round(ms2 / layers * 1e3, 2),
                               unique_experts=round(U2, 2),
                               hbm_gbs=round(b2 / (ms2 / layers * 1e-3) / 1e9, 1),
                               frac_hbm=round(b2 / (ms2 / layers * 1e-3) / 1e9 / pk["hbm"], 4))
        for name in ("decode1", "verify8", "verify8_w4a4"):
            # the same layers chained through the residual stream in persistent launches
            w5 = synth.WORKLOADS[name]
            st5 = stack if name == wl.name else build_stack(w5, layers, args.seed, device,
                                                            packs=packs)
            ms5, n5, _, U5, _ = measure_stack(w5, st5, max(3, args.steps // 2), 3,
                                              not args.no_graph, device)
            b5 = bytes_gateup(U5, w5.H, w5.I) + bytes_down(U5, w5.H, w5.I) + 12 * U5
            g5 = b5 / (ms5 / layers * 1e-3) / 1e9
            extra[name + "_stack"] = dict(
                tokens_per_s=round(w5.T * layers / (ms5 / 1e3), 1),
                us_per_layer=round(ms5 / layers * 1e3, 3), launches_per_step=n5,
                unique_experts=round(U5, 2), hbm_gbs=round(g5, 1),
                frac_hbm=round(g5 / pk["hbm"], 4),
                note=("moe_forward_layers: the layers chained through the residual stream "
                      "(x_{l+1} = BF16(x_l + out_l)), one PDL-chained launch per layer, the "
                      "residual sum written by each layer's combine"))
        if wl.name == "decode1" and wl.T == 1:
            # the same layers with a BF16 shared expert each (Is = I): two extra launches
            st4 = with_shared(stack, wl, args.seed, device)
            ms4, n4, _, _ = measure(wl, st4, max(3, args.steps // 2), 3, not args.no_graph, device)
            b4 = layer_bytes + bytes_shared(wl.H, wl.I)
            extra["decode1_shared"] = dict(
                tokens_per_s=round(wl.T * layers / (ms4 / 1e3), 1),
                us_per_layer=round(ms4 / layers * 1e3, 2), launches_per_layer=n4 // layers,
                hbm_gbs=round(b4 / (ms4 / layers * 1e-3) / 1e9, 1),
                frac_hbm=round(b4 / (ms4 / layers * 1e-3) / 1e9 / pk["hbm"], 4),
                note="routed experts' bytes + the shared expert's BF16 bytes per layer time")
            del st4
        for mode, shared in ((1, False), (0, False), (1, True), (2, False)):
            name = "prefill8192"
            w3 = synth.Workload(name, 8192, wl.H, wl.E, wl.k, wl.I, mode, 1, True)
            st3 = build_stack(w3, 1, args.seed, device, packs=packs[:1])
            if shared:
                st3 = with_shared(st3, w3, args.seed, device)
            ms3, _, _, _ = measure(w3, st3, 3, 2, False, device)
            kern3 = launch_times(w3, st3, reps=2, device=device)
            flops = 2 * w3.T * w3.k * 3 * w3.I * w3.H
            key = f"prefill8192_{['w4a16', 'w4a4', 'w4a8'][mode]}" + ("_shared" if shared else "")
            extra[key] = dict(
                tokens_per_s=round(w3.T / (ms3 / 1e3), 1), ms=round(ms3, 3),
                expert_tflops=round(flops / (ms3 * 1e-3) / 1e12, 2),
                unique_experts=st3[0].U,
                roofline=prefill_roofline(w3, ms3, kern3, st3[0].U, pk, shared),
                note=("tcgen05 block-scaled FP4 grouped GEMMs" if mode == 1 else
                      "tcgen05 kind::f16 grouped GEMMs, weights dequantised to f16 in shared "
                      "memory" + (", E4M3 activations decoded to f16" if mode == 2 else "")))
            if shared:
                sflops = 2 * w3.T * 3 * w3.I * w3.H
                extra[key].update(shared_tflop=round(sflops / 1e12, 4), note=(
                    "as prefill8192_w4a4, plus the BF16 shared expert (Is = I) on two tcgen05 "
                    "BF16 GEMMs; expert_tflops counts the routed FLOPs only"))
        torch.cuda.synchronize()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        cpu = time_oracle(wl, args.seed, 10, budget_s=25, threads=threads, n_tokens=4)

    if rank != 0:
        return
    line = dict(
        metric=METRIC, value=round(value, 2), unit="layer-tokens/s", n_gpus=world,
        steps=args.steps, warmup=args.warmup, ms_per_step=round(ms, 5), higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="nvfp4 weights, bf16/f16 operands, f32 accum",
        data="synthetic", impl="native",
        config=bench_config(wl, layers, world, args), setup_s=round(setup_s, 1),
        gpu_launches=launches * args.steps,
        roofline=roofline,
        layer=dict(us=round(ms / layers * 1e3, 3), launches=launches // layers,
                   kernel_us=None if kern is None else [(n, round(t * 1e3, 2)) for n, t in kern],
                   hbm_gbs=round(layer_gbs, 1),
                   frac_hbm=round(layer_gbs / pk["hbm"], 4), unique_experts=U_mean,
                   note=("hbm_gbs: selected experts' bytes (U x B_e)"
                         + (" + the shared expert's BF16 bytes" if args.shared else "")
                         + " per layer time, router excluded")),
        e2e=dict(value=round(world * tokens_per_step / (e2e_ms / 1e3), 2), unit="layer-tokens/s",
                 h2d_bytes_per_step=io_bytes, d2h_bytes_per_step=io_bytes,
                 graph=not args.no_graph,
                 no_graph_value=round(world * tokens_per_step / (e2e_ng_ms / 1e3), 2),
                 note=("value: the step's calls replayed from a CUDA graph between the copies; "
                       "no_graph_value: every call issued from the host (argument checks, "
                       "launch) inside the timed region")),
        clocks=clk, cpu_baseline=cpu, secondary=extra)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "native":
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_native(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
