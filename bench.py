#!/usr/bin/env python
"""Benchmark of the ternary-weight linear layer on GB300.

Default workload: the 27B-class decoder stack -- 48 distinct layers, each
with the fused QKV (5120 -> 5120+1024+1024), O (5120 -> 5120), fused
gate+up (5120 -> 2x27648) and down (27648 -> 5120) projections, ternary
weights resident in HBM in the tiled layout (6.2 GB), one token per step
(M = 1).  A step is one pass over all 192 linears; it is captured once in a
CUDA graph and replayed.  Every linear has its own synthetic X, so the four
linears of a layer are independent problems: the step issues one
tern_linear_grouped launch per layer (`per_call` times the same step with
one launch per linear, as a chain of dependent linears would need).

Reported (one JSON line on rank 0):
  value      effective weight GB/s = algorithmic bytes / step time, where a
             linear moves N*K/4 (codes) + 2*N*K/128 (FP16 scales) +
             2*M*K (bf16 X) + 4*M*N (fp32 Y) bytes
  roofline   the dominant kernel (the streaming kernel serving one layer's
             four linears, the step's only kernel, launched for every layer
             back to back outside the graph): algorithmic bytes per launch /
             average launch duration, against the measured copy bandwidth;
             `traffic` is the DRAM bytes per launch from the committed ncu
             summary while the kernel sources are unchanged
  e2e        the same metric with the step's X copied in from pinned host
             memory and all Y copied back, inside the timed region
  legs       the other listed configurations, each with its own clock record:
             27B-class linears one by one at M = 2..16 (GB/s), the stack at
             M = 2..16 and 32..256 (grouped per layer and one call per
             linear), prefill M = 1024..4096 (TFLOP/s), the 0.6B
             embedding-model layers at M = 1, 32, 512 and the single
             1024x1024 linear at M = 1, 8
  repack     GB/s of the disk -> tiled repack of all 48 layers, one
             tern_repack_grouped launch per layer (per_call_gbs: one
             tern_repack per weight)
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample

`--impl reference` times the CPU oracle alone (the reference arm).
`--profile NAME` runs one linear of layer 0 (qkv, o, gate_up, down,
gate_up_swiglu), the repack of gate_up (repack) or layer 0's four linears
as one grouped launch (layer) `--reps` times at batch `--M` and exits: the
program the committed ncu summaries under profiles/ were captured from.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "effective weight GB/s and % of HBM peak at M=1; TFLOP/s at M=4096 (27B shapes)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def linear_bytes(M: int, N: int, K: int) -> int:
    return N * K // 4 + 2 * N * (K // 128) + 2 * M * K + 4 * M * N


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- setup

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def build_stack(wl, layers, dev, tb, torch):
    """Generate, pack (GPU) and repack (GPU) every linear of the stack.

    Returns per-(layer, linear) tiled weights and the on-disk packed copies,
    and the total time tern_repack took over all layers (CUDA events)."""
    import synth
    tiled, disk = {}, {}
    for layer in range(layers):
        for lin in wl.linears:
            t, s = synth.weights(wl, layer, lin)
            t_d = torch.from_numpy(t).to(dev)
            packed = torch.empty((lin.N, lin.K // 4), dtype=torch.uint8, device=dev)
            tb.tern_pack(t_d, lin.N, lin.K, packed)
            del t_d
            disk[(layer, lin.name)] = (packed, torch.from_numpy(s.view(np.int16)).to(dev))
    # repack every layer (disk -> tiled) into buffers allocated beforehand,
    # timed with events around the repack launches alone
    for layer in range(layers):
        for lin in wl.linears:
            tiled[(layer, lin.name)] = torch.empty(tb.tern_tiled_bytes(lin.N, lin.K), dtype=torch.uint8, device=dev)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    repack_bytes = 0
    for layer in range(layers):
        for lin in wl.linears:
            packed, sc = disk[(layer, lin.name)]
            # read disk codes + scales, write tiled codes + scales
            repack_bytes += packed.numel() + 2 * sc.numel() + tiled[(layer, lin.name)].numel()
    # one tern_repack_grouped launch per layer (its four weights) ...
    torch.cuda.synchronize()
    s0.record()
    for layer in range(layers):
        srcs = [disk[(layer, lin.name)] for lin in wl.linears]
        tb.tern_repack_grouped([p for p, _ in srcs], [c for _, c in srcs], [lin.N for lin in wl.linears],
                               [lin.K for lin in wl.linears], [tiled[(layer, lin.name)] for lin in wl.linears])
    s1.record()
    torch.cuda.synchronize()
    grouped_s = s0.elapsed_time(s1) / 1e3
    # ... and one tern_repack per weight (same results, written again)
    s0.record()
    for layer in range(layers):
        for lin in wl.linears:
            packed, sc = disk[(layer, lin.name)]
            tb.tern_repack(packed, sc, lin.N, lin.K, tiled[(layer, lin.name)])
    s1.record()
    torch.cuda.synchronize()
    return tiled, disk, repack_bytes, (grouped_s, s0.elapsed_time(s1) / 1e3)


class Step:
    """All linears of the stack at batch M, with X/Y arenas on the device.
    out_type: the outputs' element type (fp32 by default; bf16 through
    tern_linear_ex).  grouped: each layer's linears -- independent problems
    here, every one with its own synthetic X -- in one tern_linear_grouped
    call (one streaming launch for M <= 16; for larger M one activation
    conversion, one GEMM and at most one split reduction) instead of one
    call each."""

    def __init__(self, wl, layers, M, tiled, dev, tb, torch, host_copies=True, out_type=0, grouped=False):
        import synth
        self.tb, self.torch = tb, torch
        self.M = M
        self.out_type = out_type
        out_size = 4 if out_type == 0 else 2
        self.calls = []
        xs, x_off, y_off = [], 0, 0
        plan = []
        for layer in range(layers):
            for lin in wl.linears:
                x = synth.activations(wl, layer, lin, M)
                xs.append(x.reshape(-1))
                plan.append((layer, lin, x_off, y_off))
                x_off += x.size
                y_off += M * lin.N
        x_host = torch.from_numpy(np.concatenate(xs).view(np.int16))
        self.x_host = x_host.pin_memory() if host_copies else None
        self.x_dev = x_host.to(dev)
        self.y_dev = torch.zeros(y_off, dtype=torch.float32 if out_type == 0 else torch.bfloat16, device=dev)
        self.y_host = torch.empty(y_off, dtype=torch.float32).pin_memory() if host_copies else None
        ws_need = 0
        self.bytes = 0
        self.flops = 0
        for layer, lin, xo, yo in plan:
            ws_need = max(ws_need, tb.tern_workspace_bytes(M, lin.N, lin.K))
            self.bytes += linear_bytes(M, lin.N, lin.K) - (4 - out_size) * M * lin.N
            self.flops += 2 * M * lin.N * lin.K
        self.grouped = grouped
        if self.grouped:
            ws_need = max(ws_need, tb.tern_grouped_workspace_bytes(M, [l.N for l in wl.linears],
                                                                   [l.K for l in wl.linears]))
        self.ws = torch.zeros(max(ws_need, 256), dtype=torch.uint8, device=dev)
        self.ws_bytes = ws_need
        for layer, lin, xo, yo in plan:
            X = self.x_dev.data_ptr() + 2 * xo
            Yp = self.y_dev.data_ptr() + out_size * yo
            self.calls.append((lin, X, tiled[(layer, lin.name)], Yp))
        self.launches_per_call = 1
        self.groups = []
        if self.grouped:
            per = len(wl.linears)
            for i in range(0, len(self.calls), per):
                cs = self.calls[i:i + per]
                self.groups.append(([c[1] for c in cs], [c[2] for c in cs], [c[0].N for c in cs],
                                    [c[0].K for c in cs], [c[3] for c in cs]))

    def run_call(self, call, stream=None):
        tb, M = self.tb, self.M
        lin, X, tl, Yp = call
        if self.out_type != 0:
            ys, off = [], 0
            for n in lin.splits:
                ys.append(Yp + 2 * M * off)
                off += n
            tb.tern_linear_ex(X, tb.TERN_X_BF16, lin.K, tl, M, lin.K, list(lin.splits), ys, list(lin.splits),
                              self.out_type, self.ws, self.ws_bytes, stream)
        elif len(lin.splits) == 1:
            tb.tern_linear(X, lin.K, tl, M, lin.N, lin.K, Yp, lin.N, self.ws, self.ws_bytes, stream)
        else:
            ys, off = [], 0
            for n in lin.splits:
                ys.append(Yp + 4 * M * off)
                off += n
            tb.tern_linear_multi(X, lin.K, tl, M, lin.K, list(lin.splits), ys, list(lin.splits),
                                 self.ws, self.ws_bytes, stream)

    def run(self, stream=None):
        if self.grouped:
            tb = self.tb
            for Xs, Ws, Ns, Ks, Ys in self.groups:
                tb.tern_linear_grouped(tb.TERN_X_BF16, self.M, Xs, Ks, Ws, Ns, Ks, Ys, Ns, self.out_type, self.ws,
                                       self.ws_bytes, stream)
            return
        for call in self.calls:
            self.run_call(call, stream)

    @property
    def launches(self):
        if self.grouped:
            return len(self.groups)
        return len(self.calls) * self.launches_per_call


def time_graph(torch, graph, steps, warmup, world, before=None, after=None, stream=None):
    for _ in range(warmup):
        if before:
            before()
        graph.replay()
        if after:
            after()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream() if stream is None else stream
    e0.record(cur)
    for _ in range(steps):
        if before:
            before()
        graph.replay()
        if after:
            after()
    e1.record(cur)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(torch, ms, world, "cuda")


def max_over_ranks(torch, value: float, world: int, device: str) -> float:
    """The slowest replica's time: every rank gets the maximum over ranks."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def capture(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()       # warm-up outside capture (sets kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        fn()
    torch.cuda.synchronize()
    return g


# --------------------------------------------------------- CPU oracle leg

def oracle_sample(wl, layers_target_s: float, M: int = 1, max_layers: int = 6):
    """Time the fp64 oracle over whole layers of the workload at batch M (up
    to `max_layers` distinct layers, passed over again) until about
    `layers_target_s` seconds of oracle time have accumulated.
    Returns (GB/s, cores, description, seconds)."""
    import oracle
    import synth
    prepared = []
    total_bytes, total_s, done = 0, 0.0, 0
    for layer in range(max_layers):
        for lin in wl.linears:
            t, s = synth.weights(wl, layer, lin)
            packed, _ = oracle.pack(t)
            del t
            prepared.append((lin, packed, s, synth.activations(wl, layer, lin, M)))
        lins = prepared[-len(wl.linears):]
        t0 = time.perf_counter()
        for lin, packed, s, x in lins:
            oracle.linear(x, packed, s, lin.K)
        total_s += time.perf_counter() - t0
        total_bytes += sum(linear_bytes(M, lin.N, lin.K) for lin, *_ in lins)
        done += 1
        if total_s >= layers_target_s:
            break
    passes = 1
    while total_s < layers_target_s:
        t0 = time.perf_counter()
        for lin, packed, s, x in prepared:
            oracle.linear(x, packed, s, lin.K)
        total_s += time.perf_counter() - t0
        total_bytes += sum(linear_bytes(M, lin.N, lin.K) for lin, *_ in prepared)
        passes += 1
    desc = (f"{done} of {wl.layers} layers ({4 * done} linears) of {wl.name} at M={M}"
            + (f", {passes} passes over them" if passes > 1 else ""))
    return total_bytes / total_s / 1e9, oracle.num_threads(), desc, total_s


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on the host cores.

    One step is a bounded sample of the decode workload: the first quarter of
    the output rows of each of layer 0's four linears at batch M."""
    if rank != 0:
        return
    import oracle
    import synth
    wl = synth.WORKLOADS[args.workload]
    prepared = []
    for lin in wl.linears:
        rows = lin.N // 4
        t, s = synth.weights(wl, 0, lin, rows=slice(0, rows))
        packed, _ = oracle.pack(t)
        del t
        prepared.append((lin, rows, packed, s, synth.activations(wl, 0, lin, args.M)))
    step_bytes = sum(linear_bytes(args.M, rows, lin.K) for lin, rows, *_ in prepared)

    def step():
        for lin, rows, packed, s, x in prepared:
            oracle.linear(x, packed, s, lin.K)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = step_bytes / dt / 1e9
    sample = (f"first N/4 output rows of each of {wl.name} layer 0's linears "
              f"(qkv, o, gate_up, down) at M={args.M}: {step_bytes / 1e6:.1f} MB per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: 27B-class linears, sampled rows", "M": args.M},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ legs

def traffic_from_profile(kernel_files, name="stream_layer_m1.txt"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if the kernel's sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None, "no profile"
    kv = {}
    for ln in lines:
        if ":" in ln:
            k, v = ln.split(":", 1)
            kv[k.strip()] = v.strip()
    h = hashlib.sha256()
    for f in kernel_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if kv.get("kernel_sources_sha256") != h.hexdigest():
        return None, "kernel changed since the capture"
    try:
        return int(kv["dram_bytes_per_launch"]), "profiles/" + name
    except (KeyError, ValueError):
        return None, "no traffic line"


KERNEL_FILES = ["ternary_bit_weight_gb300/csrc/tern_stream.cu", "ternary_bit_weight_gb300/csrc/tern_common.cuh",
                "ternary_bit_weight_gb300/csrc/tern_sm100.cuh"]


def timed_region(torch, fn, reps, local, min_ms=300.0):
    """Run fn() reps times between CUDA events on the current stream (repeating
    the batch until at least min_ms have elapsed) while sampling clocks;
    returns (ms per fn call, clocks)."""
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    total_ms, calls = 0.0, 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    while total_ms < min_ms or calls == 0:
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        total_ms += e0.elapsed_time(e1)
        calls += reps
    clocks = sampler.stop()
    return total_ms / calls, clocks


def leg_stack_batched(wl, layers, tiled, dev, tb, torch, Ms, local):
    """27B-class stack at continuous-batching sizes: tokens/s per step, with
    each layer's four linears as one grouped call (as the M = 1 headline) and
    with one call per linear (per_call)."""
    out = {}
    for M in Ms:
        row = {}
        for grouped in (True, False):
            st = Step(wl, layers, M, tiled, dev, tb, torch, host_copies=False, grouped=grouped)
            g = capture(torch, st.run)
            for _ in range(2):
                g.replay()
            ms, clocks = timed_region(torch, g.replay, 2, local, min_ms=200.0)
            r = {"ms_per_step": ms, "tokens_per_s": M / (ms / 1e3),
                 "weight_gbs": st.bytes / (ms / 1e3) / 1e9, "tflops": st.flops / (ms / 1e3) / 1e12,
                 "clocks": clocks}
            if grouped:
                row.update(r)
            else:
                row["per_call"] = r
            del g, st
            torch.cuda.empty_cache()
        out[str(M)] = row
    return out


def leg_per_linear(wl, layers, tiled, dev, tb, torch, Ms, local):
    """Each 27B-class linear at batch M, launched once per layer back to back
    (distinct weights: every launch streams from HBM); average per launch."""
    import synth
    out = {}
    for M in Ms:
        row = {}
        for lin in wl.linears:
            xs = [torch.from_numpy(synth.activations(wl, l, lin, M).view(np.int16)).to(dev) for l in range(layers)]
            Y = torch.empty((M, lin.N), dtype=torch.float32, device=dev)
            ws = torch.zeros(max(tb.tern_workspace_bytes(M, lin.N, lin.K), 256), dtype=torch.uint8, device=dev)
            outs = []
            off = 0
            for n in lin.splits:
                outs.append(Y.data_ptr() + 4 * M * off)
                off += n

            def one_pass():
                for l in range(layers):
                    if len(lin.splits) == 1:
                        tb.tern_linear(xs[l], lin.K, tiled[(l, lin.name)], M, lin.N, lin.K, Y, lin.N, ws)
                    else:
                        tb.tern_linear_multi(xs[l], lin.K, tiled[(l, lin.name)], M, lin.K, list(lin.splits), outs,
                                             list(lin.splits), ws)
            one_pass()
            ms, clocks = timed_region(torch, one_pass, 1, local, min_ms=100.0)
            us = ms * 1e3 / layers
            row[lin.name] = {"us": us, "gbs": linear_bytes(M, lin.N, lin.K) / (us * 1e-6) / 1e9,
                             "tflops": 2 * M * lin.N * lin.K / (us * 1e-6) / 1e12, "clocks": clocks}
            del xs, Y, ws
        out[str(M)] = row
    return out


def leg_prefill(wl, tiled, dev, tb, torch, Ms, local, out_type=0):
    """One layer's four linears at prefill batch sizes: TFLOP/s."""
    out = {}
    for M in Ms:
        st = Step(wl, 1, M, tiled, dev, tb, torch, host_copies=False, out_type=out_type)
        st.run()
        ms, clocks = timed_region(torch, st.run, 2, local, min_ms=200.0)
        out[str(M)] = {"ms": ms, "tflops": st.flops / (ms / 1e3) / 1e12, "clocks": clocks}
        del st
        torch.cuda.empty_cache()
    return out


def leg_workload(name, Ms, dev, tb, torch, local, reps=20, grouped=False):
    """A small workload end to end (its own weights): per-step time at each M,
    one call per linear; with `grouped` also each layer's linears as one
    grouped call (under "grouped")."""
    import synth
    wl = synth.WORKLOADS[name]
    tiled, disk, _, _ = build_stack(wl, wl.layers, dev, tb, torch)
    del disk
    out = {}
    for M in Ms:
        for grp in ((False, True) if grouped else (False,)):
            st = Step(wl, wl.layers, M, tiled, dev, tb, torch, host_copies=False, grouped=grp)
            g = capture(torch, st.run)
            for _ in range(3):
                g.replay()
            ms, clocks = timed_region(torch, g.replay, reps, local, min_ms=100.0)
            r = {"ms_per_step": ms, "tokens_per_s": M / (ms / 1e3),
                 "weight_gbs": st.bytes / (ms / 1e3) / 1e9, "clocks": clocks}
            if grp:
                out[str(M)]["grouped"] = r
            else:
                out[str(M)] = r
            del g, st
    del tiled
    torch.cuda.empty_cache()
    return out


def glu_weights(wl, layers, dev, tb, torch):
    """The gate+up linear of each layer in the GLU tile layout (tern_repack_glu
    from the fused on-disk tensor, gate rows then up rows)."""
    import synth
    lin = next(l for l in wl.linears if l.name == "gate_up")
    I, K = lin.splits[0], lin.K
    out = []
    for layer in range(layers):
        t, s = synth.weights(wl, layer, lin)
        t_d = torch.from_numpy(t).to(dev)
        packed = torch.empty((lin.N, K // 4), dtype=torch.uint8, device=dev)
        tb.tern_pack(t_d, lin.N, K, packed)
        del t_d
        sc = torch.from_numpy(s.view(np.int16)).to(dev)
        tiled = torch.empty(tb.tern_tiled_glu_bytes(I, K), dtype=torch.uint8, device=dev)
        tb.tern_repack_glu(packed, sc, packed.data_ptr() + I * (K // 4), sc.data_ptr() + I * (K // 128) * 2,
                           I, K, tiled)
        out.append(tiled)
    return lin, out


def leg_swiglu(wl, layers, dev, tb, torch, Ms, local):
    """Fused gate+up + SwiGLU (tern_linear_swiglu, bf16 h), one launch per
    layer back to back: GB/s of weights (+ X, h) and TFLOP/s per launch."""
    import synth
    lin, glu = glu_weights(wl, layers, dev, tb, torch)
    I, K = lin.splits[0], lin.K
    out = {}
    for M in Ms:
        xs = [torch.from_numpy(synth.activations(wl, l, lin, M).view(np.int16)).to(dev) for l in range(layers)]
        H = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(max(tb.tern_swiglu_workspace_bytes(M, I, K), 256), dtype=torch.uint8, device=dev)

        def one_pass():
            for l in range(layers):
                tb.tern_linear_swiglu(xs[l], tb.TERN_X_BF16, K, glu[l], M, I, K, H, I, tb.TERN_OUT_BF16, ws)
        one_pass()
        ms, clocks = timed_region(torch, one_pass, 1, local, min_ms=100.0)
        us = ms * 1e3 / layers
        nbytes = lin.N * K // 4 + 2 * lin.N * (K // 128) + 2 * M * K + 2 * M * I
        out[str(M)] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                       "tflops": 2 * M * lin.N * K / (us * 1e-6) / 1e12, "clocks": clocks}
        del xs, H, ws
    del glu
    torch.cuda.empty_cache()
    return out


def leg_variants(wl, layers, dev, tb, torch, local):
    """The layer's variants on the 27B-class shapes, one launch per layer back
    to back (distinct weights): INT8 group scales (tern_linear_s8) and int8
    activations (tern_quantize_x + tern_linear_i8) at M = 1 and 16 per
    linear, and zero-block skipping (tern_linear_sparse) on gate+up weights
    with half of the 128x128 units zero (structured sparsity) against the
    same weights run dense."""
    import synth
    out = {"s8": {}, "i8": {}, "sparse_gate_up": {}}
    for lin in wl.linears:
        K, N = lin.K, lin.N
        s8w, tiled = [], []
        for layer in range(layers):
            t, s = synth.weights(wl, layer, lin)
            t_d = torch.from_numpy(t).to(dev)
            packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
            tb.tern_pack(t_d, N, K, packed)
            del t_d
            sc = torch.from_numpy(s.view(np.int16)).to(dev)
            q8 = torch.empty((N, K // 128), dtype=torch.int8, device=dev)
            f = torch.empty(N, dtype=torch.float32, device=dev)
            tb.tern_quantize_scales(sc, N, K, q8, f)
            w8 = torch.empty(tb.tern_tiled_s8_bytes(N, K), dtype=torch.uint8, device=dev)
            tb.tern_repack_s8(packed, q8, f, N, K, w8)
            s8w.append(w8)
            w = torch.empty(tb.tern_tiled_bytes(N, K), dtype=torch.uint8, device=dev)
            tb.tern_repack(packed, sc, N, K, w)
            tiled.append(w)
        for M in (1, 16):
            xs = [torch.from_numpy(synth.activations(wl, l, lin, M).view(np.int16)).to(dev) for l in range(layers)]
            Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            ws = torch.zeros(max(tb.tern_workspace_bytes(M, N, K), tb.tern_i8_workspace_bytes(M, N, K), 256),
                             dtype=torch.uint8, device=dev)
            xq = torch.empty(tb.tern_xq_bytes(M, K), dtype=torch.int8, device=dev)
            a = torch.empty(M, dtype=torch.float32, device=dev)

            def pass_s8():
                for l in range(layers):
                    tb.tern_linear_s8(xs[l], tb.TERN_X_BF16, K, s8w[l], M, K, [N], [Y], [N], tb.TERN_OUT_F32, ws)

            def pass_i8():
                for l in range(layers):
                    tb.tern_quantize_x(xs[l], tb.TERN_X_BF16, K, M, K, xq, a)
                    tb.tern_linear_i8(xq, a, tiled[l], M, N, K, Y, N, tb.TERN_OUT_F32, ws)
            for name, fn, unit_bytes in (("s8", pass_s8, 4096 + 128), ("i8", pass_i8, 4096 + 256)):
                fn()
                ms, clocks = timed_region(torch, fn, 1, local, min_ms=60.0)
                us = ms * 1e3 / layers
                nbytes = ((N + 127) // 128) * (K // 128) * unit_bytes + M * K * 2 + 4 * M * N
                out[name].setdefault(str(M), {})[lin.name] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                                                              "clocks": clocks}
            del xs, Y, ws, xq, a
        del s8w, tiled
        torch.cuda.empty_cache()
    # zero-block skipping on gate+up with half of the units zero
    lin = next(l for l in wl.linears if l.name == "gate_up")
    K, N = lin.K, lin.N
    rng = np.random.default_rng(0)
    sp, flags = [], []
    for layer in range(layers):
        t, s = synth.weights(wl, layer, lin)
        R, G = (N + 127) // 128, K // 128
        keep = rng.random((R, G)) < 0.5
        t = t.reshape(R, 128, G, 128)
        t[~keep[:, None, :, None].repeat(128, 1).repeat(128, 3)] = 0
        t = t.reshape(N, K)
        t_d = torch.from_numpy(t).to(dev)
        packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
        tb.tern_pack(t_d, N, K, packed)
        del t_d
        w = torch.empty(tb.tern_tiled_bytes(N, K), dtype=torch.uint8, device=dev)
        tb.tern_repack(packed, torch.from_numpy(s.view(np.int16)).to(dev), N, K, w)
        fl = torch.empty(tb.tern_unit_count(N, K), dtype=torch.uint8, device=dev)
        tb.tern_zero_units(w, N, K, fl)
        sp.append(w)
        flags.append(fl)
    for M in (1, 1024):
        xs = [torch.from_numpy(synth.activations(wl, l, lin, M).view(np.int16)).to(dev) for l in range(layers)]
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws = torch.zeros(tb.tern_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)

        def dense():
            for l in range(layers):
                tb.tern_linear_ex(xs[l], tb.TERN_X_BF16, K, sp[l], M, K, [N], [Y], [N], tb.TERN_OUT_F32, ws)

        def sparse():
            for l in range(layers):
                tb.tern_linear_sparse(xs[l], tb.TERN_X_BF16, K, sp[l], flags[l], M, K, [N], [Y], [N],
                                      tb.TERN_OUT_F32, ws)
        row = {}
        for name, fn in (("dense", dense), ("skipping", sparse)):
            fn()
            ms, clocks = timed_region(torch, fn, 1, local, min_ms=60.0)
            row[name + "_us"] = ms * 1e3 / layers
            row[name + "_clocks"] = clocks
        row["speedup"] = row["dense_us"] / row["skipping_us"]
        out["sparse_gate_up"][str(M)] = row
        del xs, Y, ws
    del sp, flags
    torch.cuda.empty_cache()
    out["sparse_gate_up"]["note"] = "half of the 128x128 weight units zero, chosen at random per layer"
    return out


def run_profile(args):
    """A few calls of one layer-0 linear (or its repack) for an ncu capture."""
    import torch
    import synth
    from ternary_bit_weight_gb300 import binding as tb
    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS[args.workload]
    name = args.profile
    if name == "gate_up_swiglu":
        lin, glu = glu_weights(wl, 1, dev, tb, torch)
        I, K = lin.splits[0], lin.K
        X = torch.from_numpy(synth.activations(wl, 0, lin, args.M).view(np.int16)).to(dev)
        H = torch.empty((args.M, I), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(max(tb.tern_swiglu_workspace_bytes(args.M, I, K), 256), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            tb.tern_linear_swiglu(X, tb.TERN_X_BF16, K, glu[0], args.M, I, K, H, I, tb.TERN_OUT_BF16, ws)
        torch.cuda.synchronize()
        print("ok", name, args.M)
        return
    if name == "layer":
        # layer 0's four linears as one grouped launch
        Xs, Ws, Ys, Ns, Ks = [], [], [], [], []
        for lin in wl.linears:
            t, s = synth.weights(wl, 0, lin)
            t_d = torch.from_numpy(t).to(dev)
            packed = torch.empty((lin.N, lin.K // 4), dtype=torch.uint8, device=dev)
            tb.tern_pack(t_d, lin.N, lin.K, packed)
            del t_d
            tiled = torch.empty(tb.tern_tiled_bytes(lin.N, lin.K), dtype=torch.uint8, device=dev)
            tb.tern_repack(packed, torch.from_numpy(s.view(np.int16)).to(dev), lin.N, lin.K, tiled)
            Xs.append(torch.from_numpy(synth.activations(wl, 0, lin, args.M).view(np.int16)).to(dev))
            Ws.append(tiled)
            Ys.append(torch.empty((args.M, lin.N), dtype=torch.float32, device=dev))
            Ns.append(lin.N)
            Ks.append(lin.K)
        ws = torch.zeros(max(tb.tern_grouped_workspace_bytes(args.M, Ns, Ks), 256), dtype=torch.uint8, device=dev)
        for _ in range(args.reps):
            tb.tern_linear_grouped(tb.TERN_X_BF16, args.M, Xs, Ks, Ws, Ns, Ks, Ys, Ns, tb.TERN_OUT_F32, ws)
        torch.cuda.synchronize()
        print("ok layer", args.M)
        return
    lname = "gate_up" if name == "repack" else name
    lin = next(l for l in wl.linears if l.name == lname)
    t, s = synth.weights(wl, 0, lin)
    t_d = torch.from_numpy(t).to(dev)
    packed = torch.empty((lin.N, lin.K // 4), dtype=torch.uint8, device=dev)
    tb.tern_pack(t_d, lin.N, lin.K, packed)
    del t_d
    sc = torch.from_numpy(s.view(np.int16)).to(dev)
    tiled = torch.empty(tb.tern_tiled_bytes(lin.N, lin.K), dtype=torch.uint8, device=dev)
    if name == "repack":
        for _ in range(args.reps):
            tb.tern_repack(packed, sc, lin.N, lin.K, tiled)
        torch.cuda.synchronize()
        print("ok repack", lin.N, lin.K)
        return
    tb.tern_repack(packed, sc, lin.N, lin.K, tiled)
    X = torch.from_numpy(synth.activations(wl, 0, lin, args.M).view(np.int16)).to(dev)
    Y = torch.empty((args.M, lin.N), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(tb.tern_workspace_bytes(args.M, lin.N, lin.K), 256), dtype=torch.uint8, device=dev)
    ys, off = [], 0
    for n in lin.splits:
        ys.append(Y.data_ptr() + 4 * args.M * off)
        off += n
    for _ in range(args.reps):
        tb.tern_linear_multi(X, lin.K, tiled, args.M, lin.K, list(lin.splits), ys, list(lin.splits), ws)
    torch.cuda.synchronize()
    print("ok", name, args.M)


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack27b")
    ap.add_argument("--layers", type=int, default=48)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--no-legs", action="store_true", help="only the headline step")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", default=None,
                    help="run one layer-0 linear (or repack, gate_up_swiglu, layer) --reps times and exit")
    ap.add_argument("--reps", type=int, default=6)
    args = ap.parse_args()

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.profile:
        run_profile(args)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import synth
    from ternary_bit_weight_gb300 import binding as tb

    wl = synth.WORKLOADS[args.workload]
    layers = min(args.layers, wl.layers)
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()

    tiled, disk, repack_bytes, repack_s = build_stack(wl, layers, dev, tb, torch)
    del disk
    torch.cuda.empty_cache()

    # ---- headline: all linears of the stack at batch M, one CUDA graph per
    # step; each layer's linears (independent inputs) in one grouped launch
    step = Step(wl, layers, args.M, tiled, dev, tb, torch, grouped=True)
    graph = capture(torch, step.run)
    sampler = ClockSampler(local)
    sampler.start()
    ms = time_graph(torch, graph, args.steps, args.warmup, world)
    clocks = sampler.stop()
    value = step.bytes / (ms / 1e3) / 1e9 * world

    # ---- e2e: X in from pinned host memory, Y back out, inside the timed region
    cur = torch.cuda.current_stream()

    def h2d():
        step.x_dev.copy_(step.x_host, non_blocking=True)

    def d2h():
        step.y_host.copy_(step.y_dev, non_blocking=True)

    ms_e2e = time_graph(torch, graph, args.steps, args.warmup, world, before=h2d, after=d2h, stream=cur)
    e2e = {"value": step.bytes / (ms_e2e / 1e3) / 1e9 * world, "unit": "GB/s",
           "h2d_bytes_per_step": step.x_host.numel() * 2, "d2h_bytes_per_step": step.y_host.numel() * 4}
    del graph

    # ---- the same step with one launch per linear (a dependent chain of
    # linears cannot be grouped)
    step1 = Step(wl, layers, args.M, tiled, dev, tb, torch, host_copies=False)
    graph1 = capture(torch, step1.run)
    ms1 = time_graph(torch, graph1, args.steps, args.warmup, world)
    per_call = {"value": step1.bytes / (ms1 / 1e3) / 1e9 * world, "unit": "GB/s", "ms_per_step": ms1,
                "launches_per_step": step1.launches}
    del graph1, step1

    # ---- the dominant kernel: the streaming kernel serving one layer's four
    # linears (the step's only kernel), launched for every layer back to back
    # on the current stream; its average launch duration from CUDA events
    layer_bytes = step.bytes // layers
    ms_pass, _ = timed_region(torch, lambda: step.run(), 1, local, min_ms=100.0)
    avg_s = ms_pass / 1e3 / step.launches
    achieved = layer_bytes / avg_s / 1e9
    traffic, traffic_src = traffic_from_profile(KERNEL_FILES)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": peak_src + " (copy bandwidth)",
                "kernel": f"stream_kernel (tern_linear_grouped: one layer's qkv, o, gate_up, down; M={args.M})",
                "bytes_per_launch": layer_bytes, "avg_launch_us": avg_s * 1e6}
    per_lin = leg_per_linear(wl, layers, tiled, dev, tb, torch, [args.M], local)[str(args.M)]

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {layers} layers x (qkv, o, gate_up, down), 27B-class shapes",
                   "M": args.M, "tokens_per_step": args.M * world,
                   "weights_gb_per_step": step.bytes / 1e9,
                   "l2": "inputs larger than L2: 6.2 GB of weights streamed per step",
                   "parallelism": f"replicas x{world}", "graph": "one CUDA graph per step",
                   "launch": "one tern_linear_grouped launch per layer (its 4 linears)"},
        "hbm_frac": value / world / hbm_peak,
        "tokens_per_s": args.M * world / (ms / 1e3),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": step.launches * args.steps,
        "per_call": per_call,
        "clocks": clocks,
        "per_linear_M1": {k: {"us": v["us"], "gbs": v["gbs"]} for k, v in per_lin.items()},
        "repack": {"gbs": repack_bytes / repack_s[0] / 1e9, "layers": layers, "bytes": repack_bytes,
                   "ms": repack_s[0] * 1e3, "launch": "one tern_repack_grouped per layer",
                   "per_call_gbs": repack_bytes / repack_s[1] / 1e9},
    }
    del step
    torch.cuda.empty_cache()

    # ---- the other listed configurations, each with its own clock record
    if not args.no_legs and world == 1:
        legs = {}
        legs["dec27b_per_linear"] = leg_per_linear(wl, layers, tiled, dev, tb, torch, [2, 4, 8, 16], local)
        legs["stack27b_small_batch"] = leg_stack_batched(wl, layers, tiled, dev, tb, torch, [2, 4, 8, 16], local)
        legs["stack27b_batched"] = leg_stack_batched(wl, layers, tiled, dev, tb, torch, [32, 64, 128, 256], local)
        legs["prefill27b"] = leg_prefill(wl, tiled, dev, tb, torch, [1024, 2048, 4096], local)
        for v in legs["prefill27b"].values():
            v["frac_of_bf16_peak"] = v["tflops"] / bf16_peak
        legs["prefill27b_bf16_out"] = leg_prefill(wl, tiled, dev, tb, torch, [4096], local, out_type=1)
        for v in legs["prefill27b_bf16_out"].values():
            v["frac_of_bf16_peak"] = v["tflops"] / bf16_peak
        legs["swiglu27b"] = leg_swiglu(wl, min(layers, 8), dev, tb, torch, [1, 64, 1024], local)
        legs["variants27b"] = leg_variants(wl, min(layers, 8), dev, tb, torch, local)
        del tiled
        torch.cuda.empty_cache()
        legs["embed06b"] = leg_workload("embed06b", [1, 32, 512], dev, tb, torch, local, grouped=True)
        legs["single"] = leg_workload("single", [1, 8], dev, tb, torch, local, reps=200)
        legs["single"]["note"] = "one 1024x1024 linear: 0.28 MB of weights, L2-resident and launch-bound"
        out["legs"] = legs
        out["prefill"] = {"M": 4096, "tflops": legs["prefill27b"]["4096"]["tflops"],
                          "frac": legs["prefill27b"]["4096"]["tflops"] / bf16_peak, "peak_tflops": bf16_peak,
                          "peak_source": peak_src, "linears": "layer 0: qkv, o, gate_up, down"}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0 only)
    if rank == 0 and not args.no_cpu and world == 1:
        gbs, cores, desc, secs = oracle_sample(wl, args.cpu_seconds, M=args.M)
        out["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": secs}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
