#!/usr/bin/env python
"""Benchmark of the ternary-weight linear layer on GB300.

Default workload: the 27B-class decoder stack -- 48 distinct layers, each
with the fused QKV (5120 -> 5120+1024+1024), O (5120 -> 5120), fused
gate+up (5120 -> 2x27648) and down (27648 -> 5120) projections, ternary
weights resident in HBM in the tiled layout (6.2 GB), one token per step
(M = 1).  A step is one pass over all 192 linears; it is captured once in a
CUDA graph and replayed.

Reported (one JSON line on rank 0):
  value      effective weight GB/s = algorithmic bytes / step time, where a
             linear moves N*K/4 (codes) + 2*N*K/128 (FP16 scales) +
             2*M*K (bf16 X) + 4*M*N (fp32 Y) bytes
  roofline   the decode kernel against the measured HBM copy bandwidth
  prefill    TFLOP/s = 2*M*N*K / time at M = 4096 on one layer's linears
  repack     GB/s of tern_repack over all 48 layers (disk -> tiled)
  e2e        the same metric with the step's X copied in from pinned host
             memory and all Y copied back, inside the timed region
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample

`--impl reference` times the CPU oracle alone (the reference arm).
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
    # repack every layer (disk -> tiled), timed with events
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    repack_bytes = 0
    torch.cuda.synchronize()
    s0.record()
    for layer in range(layers):
        for lin in wl.linears:
            packed, sc = disk[(layer, lin.name)]
            out = torch.empty(tb.tern_tiled_bytes(lin.N, lin.K), dtype=torch.uint8, device=dev)
            tb.tern_repack(packed, sc, lin.N, lin.K, out)
            tiled[(layer, lin.name)] = out
            # read disk codes + scales, write tiled codes + scales
            repack_bytes += packed.numel() + 2 * sc.numel() + out.numel()
    s1.record()
    torch.cuda.synchronize()
    return tiled, disk, repack_bytes, s0.elapsed_time(s1) / 1e3


class Step:
    """All linears of the stack at batch M, with X/Y arenas on the device."""

    def __init__(self, wl, layers, M, tiled, dev, tb, torch):
        import synth
        self.tb, self.torch = tb, torch
        self.M = M
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
        self.x_host = torch.from_numpy(np.concatenate(xs).view(np.int16)).pin_memory()
        self.x_dev = self.x_host.to(dev)
        self.y_dev = torch.zeros(y_off, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(y_off, dtype=torch.float32).pin_memory()
        ws_need = 0
        self.bytes = 0
        self.flops = 0
        for layer, lin, xo, yo in plan:
            ws_need = max(ws_need, tb.tern_workspace_bytes(M, lin.N, lin.K))
            self.bytes += linear_bytes(M, lin.N, lin.K)
            self.flops += 2 * M * lin.N * lin.K
        self.ws = torch.zeros(max(ws_need, 256), dtype=torch.uint8, device=dev)
        self.ws_bytes = ws_need
        for layer, lin, xo, yo in plan:
            X = self.x_dev.data_ptr() + 2 * xo
            Yp = self.y_dev.data_ptr() + 4 * yo
            self.calls.append((lin, X, tiled[(layer, lin.name)], Yp))
        self.launches_per_call = 1

    def run_call(self, call, stream=None):
        tb, M = self.tb, self.M
        lin, X, tl, Yp = call
        if len(lin.splits) == 1:
            tb.tern_linear(X, lin.K, tl, M, lin.N, lin.K, Yp, lin.N, self.ws, self.ws_bytes, stream)
        else:
            ys, off = [], 0
            for n in lin.splits:
                ys.append(Yp + 4 * M * off)
                off += n
            tb.tern_linear_multi(X, lin.K, tl, M, lin.K, list(lin.splits), ys, list(lin.splits),
                                 self.ws, self.ws_bytes, stream)

    def run(self, stream=None):
        for call in self.calls:
            self.run_call(call, stream)

    @property
    def launches(self):
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
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms


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
    """Time the fp64 oracle over whole layers of the workload at batch M
    until about `layers_target_s` seconds of oracle time have accumulated.
    Returns (GB/s, cores, description)."""
    import oracle
    import synth
    total_bytes, total_s, done = 0, 0.0, 0
    for layer in range(max_layers):
        for lin in wl.linears:
            t, s = synth.weights(wl, layer, lin)
            packed, _ = oracle.pack(t)
            del t
            x = synth.activations(wl, layer, lin, M)
            t0 = time.perf_counter()
            oracle.linear(x, packed, s, lin.K)
            total_s += time.perf_counter() - t0
            total_bytes += linear_bytes(M, lin.N, lin.K)
        done += 1
        if total_s >= layers_target_s:
            break
    desc = f"{done} of {wl.layers} layers ({4 * done} linears) of {wl.name} at M={M}"
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
    ap.add_argument("--prefill-M", type=int, default=4096)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
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

    # ---- decode step: all linears at batch M, graph-captured
    step = Step(wl, layers, args.M, tiled, dev, tb, torch)
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

    # ---- per-linear breakdown (event-timed, not graphed): where the time goes
    per_linear = {}
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in step.calls]
    torch.cuda.synchronize()
    for call, (a, b) in zip(step.calls, ev):
        a.record()
        step.run_call(call)
        b.record()
    torch.cuda.synchronize()
    for (lin, *_), (a, b) in zip(step.calls, ev):
        per_linear.setdefault(lin.name, []).append(a.elapsed_time(b) * 1e3)
    per_linear_us = {k: statistics.median(v) for k, v in per_linear.items()}
    per_linear_gbs = {lin.name: linear_bytes(args.M, lin.N, lin.K) / (per_linear_us[lin.name] * 1e-6) / 1e9
                      for lin in wl.linears}

    # roofline of the dominant kernel: the decode kernel is every launch of the
    # step, so its average launch duration in the timed region is step/launches
    avg_launch_s = ms / 1e3 / step.launches
    achieved = step.bytes / step.launches / avg_launch_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": None, "peak_source": peak_src,
                "kernel": "umma_kernel<16> (tern_linear / tern_linear_multi, M<=16)"}

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{wl.name}: {layers} layers x (qkv, o, gate_up, down), 27B-class shapes",
                   "M": args.M, "tokens_per_step": args.M * world,
                   "weights_gb_per_step": step.bytes / 1e9,
                   "l2": "inputs larger than L2: 6.2 GB of weights streamed per step",
                   "parallelism": f"replicas x{world}", "graph": "one CUDA graph per step"},
        "hbm_frac": value / world / hbm_peak,
        "tokens_per_s": args.M * world / (ms / 1e3),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": step.launches * args.steps,
        "clocks": clocks,
        "per_linear_us": per_linear_us,
        "per_linear_gbs": per_linear_gbs,
        "repack": {"gbs": repack_bytes / repack_s / 1e9, "layers": layers,
                   "bytes": repack_bytes, "ms": repack_s * 1e3},
    }

    # ---- prefill: one layer's linears at M = prefill_M
    if not args.no_prefill:
        del graph
        pstep = Step(wl, 1, args.prefill_M, tiled, dev, tb, torch)
        pstep.run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        e0.record()
        for _ in range(reps):
            pstep.run()
        e1.record()
        torch.cuda.synchronize()
        pms = e0.elapsed_time(e1) / reps
        tflops = pstep.flops / (pms / 1e3) / 1e12
        out["prefill"] = {"M": args.prefill_M, "ms": pms, "tflops": tflops,
                          "frac": tflops / bf16_peak, "peak_tflops": bf16_peak,
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
