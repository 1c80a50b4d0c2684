#!/usr/bin/env python3
"""Benchmark of the SMOE routed-expert MoE layer forward on GB300.

Default workload: the Qwen3-235B-like decode (d_model 4096, expert ffn_dim
1536, 128 experts, top-8, renormalised), all 94 MoE layers resident in HBM
at SMOE-Q4 (120.6 GB), batch-1 decode.  One step = one token through all 94
layers in order (each layer its own seeded bf16 activation, layers
serialised on one stream, one CUDA graph per step).  `value` is decode
tokens/s.  The same measurement on the DeepSeek-MoE-16B-like layer (27
resident layers) at SMOE-Q4 and SMOE-Q2 is reported under "deepseek16b".
Weights are synthetic (seeded N(0, 0.02) with 1 % x10 outliers), generated
and grid-search quantised on the device at setup.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload qwen235b|deepseek16b|a3b35b|tiny|qwen235b_batched|...]
                    [--tokens T] [--bits 4|2|both|mixed]

The timed region is K steps bracketed by events; it is repeated until at
least a second has passed (so that the clock sampler sees it) and the median
repetition is reported.  The CPU oracle (the plain scalar C implementation
the tests check against) checks the GPU output of spot-check layers and is
timed on them, on one core and on every host core.  With --impl reference
that oracle is the whole arm, on a bounded sample of the same workload.
Under torchrun each rank runs an independent replica (the layer forward does
not shard here); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_expert_weight_gb300 import synth as Y  # noqa: E402

METRIC = "MoE-layer tokens/s and fused-dequant HBM GB/s vs GB300 peak (Q4 and Q2)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="qwen235b", choices=sorted(Y.WORKLOADS))
    p.add_argument("--tokens", type=int, default=None)
    p.add_argument("--bits", default="both", choices=["4", "2", "both", "mixed"],
                   help="mixed: the most popular quarter of the experts at Q4, the rest at Q2 "
                        "(shared expert Q4)")
    p.add_argument("--layers", type=int, default=None, help="override resident layer count")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the DeepSeek-like Q4/Q2 lines added to the default workload")
    p.add_argument("--min-timed-s", type=float, default=1.0,
                   help="repeat the K-step timed region until this much time has passed")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s: the measured burst figure (a kernel
    timed by itself), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), "measured (burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_code(text):
    """CUDA source with its comments and layout removed: what the compiler
    sees, so that a comment edit does not retire a traffic measurement."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(files=("layer.cu", "common.cuh")):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "bit_expert_weight_gb300", "csrc", f)) as fh:
            h.update(kernel_code(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, bits):
    """Per-launch DRAM bytes of the gate/up kernel from the committed ncu
    summary, or None when absent or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#"):
                if parts[0] == workload and parts[1] == f"q{bits}" and parts[3] == src:
                    return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ device model

def depths(wl, bits):
    """(per-expert depths, shared-expert depth) of a run at `bits` (2, 4 or
    "mixed": the most popular quarter of the experts by Zipf rank at Q4, the
    others at Q2, the shared expert at Q4)."""
    if bits == "mixed":
        return wl.mixed_bits(0.25), 4
    return [bits] * wl.E, bits


def expert_bytes(wl, f, bits, n_mats):
    """Codes and scales of n_mats [f, d] matrices at one depth."""
    return n_mats * (f * wl.d * bits // 8 + f * wl.d // 64 * 2)


class DeviceModel:
    """All resident layers of one workload at one bit depth, built on device:
    seeded bf16 weights (device twin of the host generator) -> grid-search
    quantiser -> repack into the tile bank."""

    def __init__(self, wl, bits, n_layers, T, dev):
        import torch

        import bit_expert_weight_gb300.smoe as S
        self.wl, self.bits, self.T, self.dev = wl, bits, T, dev
        d, f, E = wl.d, wl.f, wl.E
        self.expert_bits, self.shared_bits = depths(wl, bits)
        mixed = bits == "mixed"
        fmax = max(f, wl.shared_f)
        tmp = torch.empty(d * fmax, dtype=torch.int16, device=dev)
        self.layers, self.x, self.y = [], [], []
        t0 = time.time()
        for l in range(n_layers):
            codes, scales = [], []
            for e in range(E):
                for role in (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN):
                    rows, cols = (f, d) if role != Y.ROLE_DOWN else (d, f)
                    w = tmp[: rows * cols]
                    S.synth_bf16(w, Y.stream_key(wl.seed, l, e, role), wl.sigma, wl.p_out, 10.0,
                                 wl.p_zero)
                    c, s = S.quantize(w.view(torch.bfloat16).view(rows, cols),
                                      self.expert_bits[e])
                    codes.append(c)
                    scales.append(s)
            if mixed:
                bank = S.repack_mixed(codes, scales, d, f, self.expert_bits)
            else:
                bank = S.repack(codes, scales, d, f, E, bits)
            del codes, scales
            sh_tiles, sh_gate = None, None
            if wl.shared_f:
                sc, ss = [], []
                for role in (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN):
                    rows, cols = (wl.shared_f, d) if role != Y.ROLE_DOWN else (d, wl.shared_f)
                    w = tmp[: rows * cols]
                    S.synth_bf16(w, Y.stream_key(wl.seed, l, Y.SHARED_EXPERT, role), wl.sigma,
                                 wl.p_out, 10.0, wl.p_zero)
                    c, s = S.quantize(w.view(torch.bfloat16).view(rows, cols),
                                      self.shared_bits)
                    sc.append(c)
                    ss.append(s)
                sh_tiles = S.repack(sc, ss, d, wl.shared_f, 1, self.shared_bits)
                if wl.shared_gate:
                    sh_gate = torch.from_numpy(wl.shared_gate_weight(l).view(np.int16)).to(
                        dev).view(torch.bfloat16)
            router = torch.from_numpy(wl.router_weight(l).view(np.int16)).to(dev).view(
                torch.bfloat16)
            # the batched workload's Zipf(s) popularity as a selection-only bias
            bias = None
            if wl.zipf_s:
                bias = torch.from_numpy(wl.zipf_bias()).to(dev)
            self.layers.append(S.MoELayer(d, f, E, wl.k, wl.norm, self.shared_bits, router, bank,
                                          expert_bias=bias, shared_tiles=sh_tiles,
                                          shared_f=wl.shared_f, shared_gate_w=sh_gate,
                                          expert_bits=self.expert_bits if mixed else None))
        # every layer's tokens and outputs in one contiguous tensor each, so
        # that a step's inputs and results cross PCIe/C2C in one copy each
        xdt = torch.bfloat16 if wl.x_dtype == "bf16" else torch.float32
        self.x_all = torch.empty((n_layers, T, d), dtype=xdt, device=dev)
        self.y_all = torch.empty((n_layers, T, d), dtype=torch.float32, device=dev)
        for l in range(n_layers):
            xf, xb = wl.activations(l, T)
            if xb is not None:
                self.x_all[l].view(torch.int16).copy_(torch.from_numpy(xb.view(np.int16)))
            else:
                self.x_all[l].copy_(torch.from_numpy(xf))
        self.x = [self.x_all[l] for l in range(n_layers)]
        self.y = [self.y_all[l] for l in range(n_layers)]
        torch.cuda.synchronize()
        self.setup_s = time.time() - t0
        self.ws = S.workspace(self.layers[0], T)
        self.grouped = S.path_for(self.layers[0], T) == S.PATH_GROUPED
        self.ids = [torch.empty((T, wl.k), dtype=torch.int32, device=dev) for _ in self.layers]
        self.resident_bytes = sum(l.expert_tiles.numel() for l in self.layers)

    def step(self):
        import bit_expert_weight_gb300.smoe as S
        for lay, x, y, ids in zip(self.layers, self.x, self.y, self.ids):
            S.forward(lay, x, self.ws, y=y, ids=ids)

    def step_timed(self, evs):
        """The same step with events around the dominant kernel of every
        layer: for T <= 8 the fused layer kernel (router, experts, combine);
        on the grouped path the gate/up grouped GEMM (stage 1), the other
        stages bracketed by events too (evs[i] = 4 events)."""
        import bit_expert_weight_gb300.smoe as S
        for i, (lay, x, y, ids) in enumerate(zip(self.layers, self.x, self.y, self.ids)):
            if self.grouped:
                evs[i][2].record()
                S.forward_stage(lay, 0, x, self.ws, y, ids=ids)
                evs[i][0].record()
                S.forward_stage(lay, 1, x, self.ws, y, ids=ids)
                evs[i][1].record()
                S.forward_stage(lay, 2, x, self.ws, y, ids=ids)
                evs[i][3].record()
            else:
                evs[i][0].record()
                S.forward(lay, x, self.ws, y=y, ids=ids)
                evs[i][1].record()


def layer_algorithmic_bytes(model):
    """Whole-layer algorithmic bytes (router + distinct experts' gate/up/down
    codes and scales + x + y), averaged over layers."""
    wl = model.wl
    tot = 0
    for ids in model.ids:
        b = sum(expert_bytes(wl, wl.f, model.expert_bits[e], 3) for e in np.unique(ids.cpu().numpy()))
        b += wl.E * wl.d * 2 + model.T * wl.d * (model.x[0].element_size() + 4)
        if wl.shared_f:
            b += expert_bytes(wl, wl.shared_f, model.shared_bits, 3) + wl.d * 2
        tot += b
    return tot / len(model.ids)


def gateup_bytes(model):
    """Algorithmic bytes of the gate/up grouped GEMM per layer: the gate and
    up codes and scales of the distinct experts the tokens selected (plus the
    shared expert's), the bf16 token rows in and the bf16 h rows out."""
    wl = model.wl
    b = np.mean([sum(expert_bytes(wl, wl.f, model.expert_bits[e], 2)
                     for e in np.unique(ids.cpu().numpy())) for ids in model.ids])
    b += model.T * wl.d * 2 + model.T * wl.k * wl.f * 2
    if wl.shared_f:
        b += expert_bytes(wl, wl.shared_f, model.shared_bits, 2)
        b += model.T * wl.shared_f * 2
    return float(b)


def gateup_flops(model):
    """Algorithmic flops of the gate/up grouped GEMM per layer: 2 (gate and
    up) x 2 (multiply-add) x d x f per routed (token, slot), plus the shared
    expert's over all tokens; padding rows are not counted."""
    wl = model.wl
    f = 4.0 * model.T * wl.k * wl.d * wl.f
    if wl.shared_f:
        f += 4.0 * model.T * wl.d * wl.shared_f
    return f


def max_over_ranks(value, world, dev):
    """The largest of every rank's value (all ranks call it; world 1: the
    value itself).  The timed region ends when the slowest replica does."""
    import torch
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def launches_per_layer(model):
    """Kernels one layer forward launches: the fused layer kernel for T <= 8
    on the streaming path, else router + layer + combine; on the grouped path
    router (bf16: logits GEMM + routing), sort, gather, one gate/up and one
    down GEMM per depth present, combine."""
    if not model.grouped:
        return 1 if model.T <= 8 else 3
    router = 2 if model.x[0].dtype.itemsize == 2 else 1
    present = set(model.expert_bits) | ({model.shared_bits} if model.wl.shared_f else set())
    return router + 3 + 2 * len(present)


def run_bits(args, wl, bits, n_layers, T, dev, world, rank):
    import torch
    torch.cuda.synchronize()
    model = DeviceModel(wl, bits, n_layers, T, dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    use_graph = not args.no_graph
    with torch.cuda.stream(stream):
        model.step()  # eager warm-up + routing for the byte counts
    stream.synchronize()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            model.step()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            with torch.cuda.stream(stream):
                model.step()

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            run_step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    # K timed steps per repetition, repeated until min_timed_s has passed on
    # the host clock (at least once); every repetition is bracketed by a
    # barrier and a synchronize, and its length is the slowest rank's
    rep_ms = []
    t_start = time.perf_counter()
    while not rep_ms or time.perf_counter() - t_start < args.min_timed_s:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(args.steps):
                run_step()
            e1.record()
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        rep_ms.append(max_over_ranks(e0.elapsed_time(e1), world, dev))
    clocks = clk.stop()
    ms = float(np.median(rep_ms))
    ms_per_step = ms / args.steps
    tok_s = world * T * args.steps / (ms / 1e3)

    # dominant kernel (the fused layer kernel): events around each launch
    reps = max(3, min(50, args.steps))
    evs = [tuple(torch.cuda.Event(enable_timing=True, external=True) for _ in range(4))
           for _ in model.layers]
    g2 = None
    if use_graph:
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            model.step_timed(evs)
    durs, stage_ms = [], []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            if g2 is not None:
                g2.replay()
            else:
                model.step_timed(evs)
            stream.synchronize()
            durs.extend(e[0].elapsed_time(e[1]) for e in evs)
            if model.grouped:
                stage_ms.extend((e[2].elapsed_time(e[0]), e[0].elapsed_time(e[1]),
                                 e[1].elapsed_time(e[3])) for e in evs)
    kern_ms = float(np.mean(durs))
    layer_bytes = layer_algorithmic_bytes(model)

    # end to end: pinned host x -> device, forward, device y -> host, per step
    # (all layers' tokens in one copy, all their outputs in one copy)
    x_host = model.x_all.cpu().pin_memory()
    y_host = torch.empty_like(model.y_all, device="cpu").pin_memory()
    h2d = x_host.numel() * x_host.element_size()
    d2h = y_host.numel() * y_host.element_size()

    def e2e_step():
        model.x_all.copy_(x_host, non_blocking=True)
        model.step()
        y_host.copy_(model.y_all, non_blocking=True)

    g3 = None
    if use_graph:
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=stream):
            e2e_step()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g3.replay() if g3 is not None else e2e_step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record()
        for _ in range(args.steps):
            g3.replay() if g3 is not None else e2e_step()
        f1.record()
    stream.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev)
    import bit_expert_weight_gb300.smoe as S
    status = S.device_status(stream)
    res = {
        "bits": bits, "tokens_per_s": tok_s, "ms_per_step": ms_per_step,
        "layer_tokens_per_s": tok_s * n_layers, "layers": n_layers, "T": T,
        "layer_us": ms_per_step * 1e3 / n_layers,
        "layer_alg_bytes": layer_bytes,
        "layer_alg_GBps": layer_bytes / (ms_per_step * 1e-3 / n_layers) / 1e9,
        "kernel_us": kern_ms * 1e3,
        "kernel_alg_GBps": layer_bytes / (kern_ms * 1e-3) / 1e9,
        "e2e_tokens_per_s": world * T * args.steps / (e2e_ms / 1e3),
        "h2d": h2d, "d2h": d2h, "clocks": clocks, "setup_s": model.setup_s,
        "resident_GB": model.resident_bytes / 1e9, "device_status": status,
        "launches_per_step": n_layers * launches_per_layer(model),
        "grouped": model.grouped,
        "stage_us": [float(v) * 1e3 for v in np.mean(stage_ms, axis=0)] if stage_ms else None,
        "expert_bits": list(model.expert_bits), "shared_bits": model.shared_bits,
        "gemm1_flops": gateup_flops(model) if model.grouped else None,
        "gemm1_bytes": gateup_bytes(model) if model.grouped else None,
        "y_layers": {l: model.y[l].float().cpu().numpy() for l in check_layers(n_layers)},
        "timed_reps": len(rep_ms), "rep_ms": rep_ms,
        "routing": routing_summary([i.cpu().numpy() for i in model.ids], wl, list(model.expert_bits),
                                   model.shared_bits),
    }
    del model, graph, g2, g3
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ CPU oracle

def check_layers(n_layers):
    """Spot-check layers of a stack: four evenly spaced (0, 31, 62 and 93
    of 94), every layer of a stack of four or fewer."""
    if n_layers <= 4:
        return list(range(n_layers))
    return sorted({int(round(i * (n_layers - 1) / 3)) for i in range(4)})


def _quant_job(job):
    """Pool worker: one weight matrix from the host generator, quantised by
    the oracle."""
    import oracle as O
    wl_name, layer, e, role, bits = job
    w = Y.WORKLOADS[wl_name].expert_weight(layer, e, role)
    return O.quantize(w, bits)


def prepare_oracle(wl, bits, layers, T):
    """Per layer: seeded tokens plus the oracle-quantised blobs of exactly
    the experts those tokens select (generated on the host and quantised
    untimed, in a spawn pool)."""
    import multiprocessing as mp

    import oracle as O
    O.build_oracle()
    ebits, sbits = depths(wl, bits)
    roles = (Y.ROLE_GATE, Y.ROLE_UP, Y.ROLE_DOWN)
    name = next(k for k, v in Y.WORKLOADS.items() if v is wl)
    per_layer, jobs = [], []
    for layer in layers:
        xf, _ = wl.activations(layer, T)
        router = wl.router_weight(layer)
        bias = wl.zipf_bias() if wl.zipf_s else None
        ids, _ = O.route(O.router_logits(router, xf), wl.k, wl.norm, bias)
        experts = sorted(set(int(e) for e in ids.ravel()))
        j0 = len(jobs)
        jobs += [(name, layer, e, r, ebits[e]) for e in experts for r in roles]
        if wl.shared_f:
            jobs += [(name, layer, Y.SHARED_EXPERT, r, sbits) for r in roles]
        per_layer.append((layer, xf, router, bias, experts, j0))
    with mp.get_context("spawn").Pool(min(len(jobs), os.cpu_count() or 1)) as pool:
        qs = pool.map(_quant_job, jobs)
    preps = []
    for layer, xf, router, bias, experts, j0 in per_layer:
        blobs = {e: O.make_blob(*qs[j0 + 3 * i:j0 + 3 * i + 3]) for i, e in enumerate(experts)}
        n = j0 + 3 * len(experts)
        sb = O.make_blob(*qs[n:n + 3]) if wl.shared_f else None
        sg = wl.shared_gate_weight(layer) if wl.shared_gate else None
        preps.append({"layer": layer, "x": xf, "router": router, "blobs": blobs,
                      "shared_blob": sb, "shared_gate": sg, "bias": bias})
    return preps


def time_oracle(wl, bits, prep, nthreads=1):
    """(seconds, y) of one oracle layer forward of the prepared tokens:
    router logits, routing, then the expert FFNs and the combine -- on one
    thread, or with the (token, slot) expert FFNs spread over nthreads."""
    import oracle as O
    ebits, sbits = depths(wl, bits)
    eb = ebits if bits == "mixed" else None
    t0 = time.perf_counter()
    lg = O.router_logits(prep["router"], prep["x"])
    ids, w = O.route(lg, wl.k, wl.norm, prep["bias"])
    kw = dict(shared_blob=prep["shared_blob"], fs=wl.shared_f, shared_gate=prep["shared_gate"],
              expert_bits=eb)
    if nthreads <= 1:
        y = O.moe_apply(wl.d, wl.f, wl.E, wl.k, sbits, prep["blobs"], prep["x"], ids, w, **kw)
    else:
        y = O.moe_apply_threads(wl.d, wl.f, wl.E, wl.k, sbits, prep["blobs"], prep["x"], ids, w,
                                nthreads, **kw)
    return time.perf_counter() - t0, y


def time_oracle_layers(wl, bits, preps, nthreads, min_s):
    """Passes over the prepared layers until min_s has passed (at least one);
    returns (mean seconds per layer forward, passes, y per layer)."""
    times, ys, passes = [], {}, 0
    t_start = time.perf_counter()
    while passes == 0 or time.perf_counter() - t_start < min_s:
        for prep in preps:
            sec, y = time_oracle(wl, bits, prep, nthreads)
            times.append(sec)
            ys[prep["layer"]] = y
        passes += 1
    return float(np.mean(times)), passes, ys


def parity_summary(y_gpu, y_ref, bar):
    """Largest elementwise difference of the GPU layer output from the
    oracle's, against the path's bar (a fraction of max |y_ref|)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    err = float(np.abs(y_gpu - y_ref).max()) if y_ref.size else 0.0
    ref = float(np.abs(y_ref).max()) if y_ref.size else 0.0
    rel = err / ref if ref > 0 else 0.0
    return {"max_abs_err": err, "ref_max_abs": ref, "rel": rel, "bar": bar, "ok": rel <= bar}


def routing_summary(ids_list, wl, expert_bits, shared_bits):
    """Realised routing of a step: selections per expert summed over the
    layers, the distinct experts per layer, the busiest expert's share, and
    the expert weights the step streams (every distinct selected expert of
    every layer at its depth, plus the shared expert): the footprint that
    must exceed L2 for back-to-back steps to read HBM without a flush."""
    E = wl.E
    hist = np.zeros(E, dtype=np.int64)
    distinct = []
    step_bytes = 0
    for ids in ids_list:
        v = np.asarray(ids).ravel()
        v = v[(v >= 0) & (v < E)]
        hist += np.bincount(v, minlength=E)
        u = np.unique(v)
        distinct.append(len(u))
        step_bytes += sum(expert_bytes(wl, wl.f, expert_bits[e], 3) for e in u.tolist())
        if wl.shared_f:
            step_bytes += expert_bytes(wl, wl.shared_f, shared_bits, 3)
    total = int(hist.sum())
    return {"distinct_experts_per_layer": float(np.mean(distinct)) if distinct else 0.0,
            "max_expert_share": float(hist.max()) / total if total else 0.0,
            "weight_MB_per_step": step_bytes / 1e6,
            "l2_MB": 129,
            "histogram": hist.tolist()}


def host_cores():
    """Host cores this process may run on (the oracle's thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def default_bits(args, wl):
    if args.bits == "mixed":
        return ["mixed"]
    if args.bits == "both":
        return [b for b in (4, 2) if b in wl.bits_list]
    return [int(args.bits)]  # an explicit depth, whatever the workload lists


def config_dict(wl, n_layers, T, bits, world, graph):
    """The line's config: the workload by name and geometry.  Computed from
    the workload alone, so that both arms print the same dict."""
    ebits, sbits = depths(wl, bits)
    bank = sum(expert_bytes(wl, wl.f, b, 3) for b in ebits)
    if wl.shared_f:
        bank += expert_bytes(wl, wl.shared_f, sbits, 3)
    return {"workload": wl.name, "layers": n_layers, "tokens_per_step": T, "bits": bits,
            "d_model": wl.d, "ffn_dim": wl.f, "experts": wl.E, "top_k": wl.k,
            "norm_topk_prob": wl.norm, "shared_ffn_dim": wl.shared_f,
            "resident_GB": round(n_layers * bank / 1e9, 3),
            "l2": "no flush: inputs larger than L2 (the realised per-step weight footprint is "
                  "routing.weight_MB_per_step, against 129 MB of L2)",
            "graph": graph, "parallelism": f"replicas x{world}"}


def run_reference(args, wl, T, n_layers, world, rank):
    """The oracle as the reference arm, on every host core: each step is the
    oracle forward of the workload's T tokens through one spot-check layer
    (cycling through them), and the step time is that layer's time times the
    layer count (tokens/s through all layers, extrapolated)."""
    if rank != 0:
        return
    bits = default_bits(args, wl)[0]
    layers = check_layers(n_layers)
    preps = prepare_oracle(wl, bits, layers, T)
    cores = host_cores()
    for i in range(args.warmup):
        time_oracle(wl, bits, preps[i % len(preps)], cores)
    per = [time_oracle(wl, bits, preps[i % len(preps)], cores)[0] for i in range(args.steps)]
    layer_s = float(np.mean(per))
    step_s = layer_s * n_layers
    v = T / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": config_dict(wl, n_layers, T, bits, world, not args.no_graph),
        "extrapolation": {"timed": f"{args.steps} oracle layer forwards of {T} token(s), "
                                   f"cycling through layers {layers}",
                          "per_step": f"x{n_layers} layers"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"oracle forward of {T} token(s) through one of layers "
                                   f"{layers} per step ({layer_s:.3f} s each on {cores} "
                                   f"threads), x{n_layers} layers extrapolated"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def side_summary(q, hbm):
    """The fields of a run reported beside the headline (another depth or
    workload)."""
    return {"value": q["tokens_per_s"], "unit": "tokens/s", "layers": q["layers"],
            "ms_per_step": q["ms_per_step"], "layer_us": q["layer_us"],
            "layer_alg_bytes": q["layer_alg_bytes"], "layer_alg_GBps": q["layer_alg_GBps"],
            "frac": q["layer_alg_GBps"] / hbm,
            "isolated_launch": {"us": q["kernel_us"], "alg_GBps": q["kernel_alg_GBps"],
                                "frac": q["kernel_alg_GBps"] / hbm},
            "e2e": q["e2e_tokens_per_s"], "clocks": q["clocks"],
            "device_status": q["device_status"], "timed_reps": q["timed_reps"]}


# ------------------------------------------------------------------ main

def main():
    args = parse()
    wl = Y.WORKLOADS[args.workload]
    T = args.tokens if args.tokens is not None else wl.T_list[0]
    n_layers = args.layers if args.layers is not None else wl.layers
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, wl, T, n_layers, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import torch
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from bit_expert_weight_gb300 import build
    build.build()
    bits_list = default_bits(args, wl)
    results = {b: run_bits(args, wl, b, n_layers, T, dev, world, rank) for b in bits_list}
    # the metric names Q4 and Q2: the default (Q4-only) workload adds the
    # DeepSeek-like stack at both depths
    extra = {}
    if args.workload == "qwen235b" and args.tokens is None and not args.no_extra:
        ds = Y.WORKLOADS["deepseek16b"]
        for b in (4, 2):
            extra[b] = run_bits(args, ds, b, ds.layers, 1, dev, world, rank)
    hbm, peak_kind = peaks()
    main_bits = bits_list[0]
    r = results[main_bits]
    traffic = ncu_traffic(args.workload, main_bits)
    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline:
        layers = check_layers(n_layers)
        preps = prepare_oracle(wl, main_bits, layers, T)
        cores = host_cores()
        s1, p1, ys = time_oracle_layers(wl, main_bits, preps, 1, 5.0)
        sn, pn, _ = time_oracle_layers(wl, main_bits, preps, cores, 5.0)
        bar = 2e-2 if r["grouped"] else 1e-3
        per = {l: parity_summary(r["y_layers"][l], ys[l], bar) for l in layers}
        worst = max(per.values(), key=lambda v: v["rel"])
        parity = dict(worst)
        parity.update({"layers": layers, "tokens": T, "ok": all(v["ok"] for v in per.values()),
                       "rel_per_layer": {str(l): v["rel"] for l, v in per.items()}})
        sample = (f"oracle forward of {T} token(s) through layers {layers} "
                  f"(mean per layer), x{n_layers} layers extrapolated")
        cpu = {"value": T / (sn * n_layers), "unit": "tokens/s", "cores": cores,
               "kind": "oracle",
               "sample": f"{sample}; {pn} passes of {sn:.3f} s per layer on {cores} threads",
               "single_core": {"value": T / (s1 * n_layers), "cores": 1,
                               "sample": f"{sample}; {p1} passes of {s1:.3f} s per layer"}}
    if rank != 0:
        return
    if r["grouped"]:
        # the binding roofline of the gate/up GEMM: flops / tensor peak or
        # weight bytes / HBM bandwidth, whichever ideal time is longer
        tp, tp_kind = tensor_peak()
        t_tc = r["gemm1_flops"] / (tp * 1e12)
        t_hbm = r["gemm1_bytes"] / (hbm * 1e9)
        sec = r["kernel_us"] * 1e-6
        if t_tc >= t_hbm:
            ach = r["gemm1_flops"] / sec / 1e12
            roofline = {"bound": "tensor", "achieved": ach, "peak": tp, "unit": "TFLOP/s",
                        "frac": ach / tp, "peak_kind": tp_kind}
        else:
            ach = r["gemm1_bytes"] / sec / 1e9
            roofline = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                        "frac": ach / hbm, "peak_kind": peak_kind}
        roofline.update({
            "traffic": None,
            "kernel": "grouped_gemm_kernel (gate/up: dequant to bf16 in shared memory, "
                      "tcgen05 MMA, SiLU(g)*u epilogue)",
            "flops_per_launch": r["gemm1_flops"], "bytes_per_launch": r["gemm1_bytes"],
            "launch_us": r["kernel_us"],
            "ideal_us": {"tensor": t_tc * 1e6, "hbm": t_hbm * 1e6},
            "stage_us": {"route_sort_gather": r["stage_us"][0],
                         "gateup_gemm": r["stage_us"][1],
                         "down_gemm_combine": r["stage_us"][2]}})
    else:
        # the layer kernel is the whole layer: its achieved bandwidth is the
        # algorithmic bytes of a step over the step time (launch gaps
        # included); the event-bracketed launch is reported beside it
        roofline = {"bound": "hbm", "achieved": r["layer_alg_GBps"], "peak": hbm,
                    "unit": "GB/s", "frac": r["layer_alg_GBps"] / hbm, "traffic": traffic,
                    "kernel": "moe_layer_kernel (router, top-k, dispatch, fused dequant "
                              "gate/up + SiLU, fused dequant down, combine)",
                    "bytes_per_launch": r["layer_alg_bytes"],
                    "basis": "algorithmic bytes x layers / ms_per_step",
                    "layer_us": r["layer_us"], "peak_kind": peak_kind,
                    "isolated_launch": {"us": r["kernel_us"], "achieved": r["kernel_alg_GBps"],
                                        "frac": r["kernel_alg_GBps"] / hbm,
                                        "note": "CUDA events around each launch (breaks the "
                                                "overlap of consecutive launches)"}}
    line = {
        "metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights + 1% x10 outliers, grid-search "
                "quantised on device; N(0,1) bf16 activations)",
        "config": config_dict(wl, n_layers, T, main_bits, world, not args.no_graph),
        "timed_reps": r["timed_reps"], "rep_ms": r["rep_ms"],
        "roofline": roofline,
        "depths": {"q4_experts": r["expert_bits"].count(4), "q2_experts": r["expert_bits"].count(2),
                   "shared": r["shared_bits"] if wl.shared_f else None},
        "layer": {"us": r["layer_us"], "alg_GBps": r["layer_alg_GBps"],
                  "frac": r["layer_alg_GBps"] / hbm, "tokens_per_s": r["layer_tokens_per_s"]},
        "e2e": {"value": r["e2e_tokens_per_s"], "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches_per_step"] * args.steps * r["timed_reps"],
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
        "setup_s": round(r["setup_s"], 1),
        "device_status": r["device_status"],
        "parity_vs_oracle": parity,
        "routing": r["routing"],
    }
    for b in bits_list[1:]:
        line[f"q{b}"] = side_summary(results[b], hbm)
    if extra:
        line["deepseek16b"] = {f"q{b}": side_summary(q, hbm) for b, q in extra.items()}
        q4, q2 = extra[4], extra[2]
        line["deepseek16b"]["q2_over_q4_layer_time"] = q2["layer_us"] / q4["layer_us"]
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
