#!/usr/bin/env python3
"""Benchmark of the K3 LatentMoE MXFP4 routed-expert layer on GB300.

Default workload: one K3-dim routed layer at decode sizes (H=7168,
L=3584, 896 experts top-16, I=3072, ~15.7 GB of MXFP4 expert weights); one
step = one forward of a fresh T=1 batch, a fresh T=8 batch and a fresh
T=64 batch (73 tokens).  Inputs and weights are seeded synthetic data and
are resident in HBM before timing.  L2 is flushed before every forward,
outside the timed events: a 512 MB write, then a 256 MB read, so that the
forward starts with no weight or input bytes in L2 and without the flush's
own dirty lines waiting to be written back.  Each forward is replayed from a
CUDA graph captured from the library's C-ABI forward call.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (a bounded sample of the same workload per step).
Under torchrun every rank runs its own replica of the workload on its own
GPU (tokens are independent: weak scaling, no data-path collective);
timing is max over ranks and `value` sums the ranks' tokens.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DECODE_BATCHES = (1, 8, 64)
PREFILL_T = 8192
METRIC = "LatentMoE MXFP4 layer tokens/s (K3 dims); decode HBM GB/s vs ~8 TB/s"
FLUSH_BYTES = 512 << 20
REASON_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
    0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
    0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
}


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def reduce_max_over_ranks(value: float, world: int, device=None) -> float:
    """max over ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms with a
    timestamp; only the samples taken inside the timed region's wall-clock
    window [begin(), end()] are kept."""

    QUERY = "timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"

    def __init__(self, gpu_index: int, settle_s: float = 1.5):
        self.proc = None
        self.t0 = self.t1 = None
        self.windows = {}
        self.window_summaries = {}
        import tempfile
        try:
            fd, self.path = tempfile.mkstemp(prefix="k3moe_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(settle_s)  # nvidia-smi needs a moment before its first sample
        except Exception:
            self.proc = None

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def mark(self, name: str, t0: float, t1: float):
        """Record a further wall-clock window (a later leg of the run) to
        summarise separately."""
        self.windows[name] = (t0, t1)

    @staticmethod
    def _stamp(text: str):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        try:
            self.window_summaries = {k: self.parse(a, b) for k, (a, b) in self.windows.items()}
            return self.parse()
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass

    def parse(self, t0=None, t1=None) -> dict:
        t0 = self.t0 if t0 is None else t0
        t1 = self.t1 if t1 is None else t1
        sm, smax, reasons, window = [], None, set(), 0
        lo = (t0 if t0 is not None else float("-inf")) - 0.02
        hi = (t1 if t1 is not None else float("inf")) + 0.02
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            ts = self._stamp(parts[0])
            try:
                clk, mx = float(parts[2]), float(parts[3])
                act = int(parts[5], 16)
            except ValueError:
                continue
            smax = mx
            if ts is None or not (lo <= ts <= hi):
                continue
            window += 1
            sm.append(clk)
            for bit, name in REASON_BITS.items():
                if act & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": window, "interval_ms": 20}


def source_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per active expert of `kernel` from a committed ncu capture
    (profiles/traffic.json), if the kernel's source is unchanged since the
    counters were taken; None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "mxfp4_routed_expert_k3_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or source_sha(src) != rec.get("source_sha"):
        return None
    return rec["dram_bytes_per_active_expert"]


# ============================================================================ ours
def run_ours(args, rank, world, local_rank):
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    from mxfp4_routed_expert_k3_gb300.dims import K3

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    d = K3 if args.experts == K3.n_experts else K3.with_(n_experts=args.experts)
    batches = DECODE_BATCHES
    maxT = max(batches)
    w = synth.layer_weights(d, seed=1)
    prefill_T = 0 if args.no_prefill else args.prefill_tokens
    layer = k3moe.Layer(d, w, max_tokens=max(maxT, prefill_T), device=local_rank, force_path=args.path)
    stream = torch.cuda.Stream(device=dev)
    pool = args.warmup + args.steps
    # fresh token batches for every step, resident in HBM before timing
    xs = {T: [torch.from_numpy(synth.token_rows(d, 5000 + 97 * rank + 13 * i + T, T).view(np.int16)).to(dev)
              for i in range(pool)] for T in batches}
    x_in = {T: torch.empty((T, d.hidden), dtype=torch.int16, device=dev) for T in batches}
    y = {T: torch.empty((T, d.hidden), dtype=torch.int16, device=dev) for T in batches}
    idx = {T: torch.empty((T, d.top_k), dtype=torch.int32, device=dev) for T in batches}
    wt = {T: torch.empty((T, d.top_k), dtype=torch.float32, device=dev) for T in batches}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(FLUSH_BYTES // 8, dtype=torch.int32, device=dev)

    def l2_flush():
        flush.zero_()      # evicts everything (512 MB > 129 MB of L2) ...
        flush_rd.sum()     # ... and reading 256 MB writes the dirty lines back

    with torch.cuda.stream(stream):
        for T in batches:  # eager warm-up before capture
            x_in[T].copy_(xs[T][0])
            layer.forward(x_in[T], y[T], idx[T], wt[T], stream=stream)
    stream.synchronize()
    # timed graphs hold the forward alone; a second set, captured with the
    # per-launch-group events, gives the kernel split after the timed region
    def capture(profiled):
        k3moe.profile(layer.ctx, profiled)
        out = {}
        for T in batches:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                layer.forward(x_in[T], y[T], idx[T], wt[T], stream=stream)
            out[T] = g
        return out
    graphs = capture(False)
    launches_per_forward = {}
    for T in batches:
        layer.forward(x_in[T], y[T], idx[T], wt[T], stream=stream)
        launches_per_forward[T] = layer.query("launches_last")
    stream.synchronize()
    # captured last and left enabled until read: an eager forward or
    # disabling the profile resets the context's record of the event slots
    graphs_prof = capture(True)

    ev = {T: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(pool)]
          for T in batches}
    per_kernel = {T: [] for T in batches}
    active_experts = {T: [] for T in batches}

    def one_step(i, record):
        for T in batches:
            with torch.cuda.stream(stream):
                l2_flush()
                x_in[T].copy_(xs[T][i])
                ev[T][i][0].record(stream)
                graphs[T].replay()
                ev[T][i][1].record(stream)
            if record:
                stream.synchronize()
                act = np.empty(d.n_experts + 1, np.int32)
                k3moe.fetch(layer.ctx, "active", act)
                active_experts[T].append(int(act[0]))

    for i in range(args.warmup):
        one_step(i, False)
    stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local_rank)
    torch.cuda.synchronize()
    clocks.begin()
    t_wall0 = time.perf_counter()
    for i in range(args.warmup, pool):
        one_step(i, True)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clocks.end()
    barrier(world)
    assert layer.status() == 0, k3moe.last_error(layer.ctx)
    # per-launch-group split: the profiled graphs on the same inputs
    for i in range(args.warmup, pool):
        for T in batches:
            with torch.cuda.stream(stream):
                l2_flush()
                x_in[T].copy_(xs[T][i])
                graphs_prof[T].replay()
            stream.synchronize()
            per_kernel[T].append(k3moe.profile_read(layer.ctx))
    k3moe.profile(layer.ctx, False)

    fwd_ms = {T: [ev[T][i][0].elapsed_time(ev[T][i][1]) for i in range(args.warmup, pool)] for T in batches}
    step_ms = sum(statistics.mean(fwd_ms[T]) for T in batches)
    tokens_per_step = sum(batches)
    step_ms_max = reduce_max_over_ranks(step_ms, world, dev)
    value = tokens_per_step * world / (step_ms_max / 1e3)

    # ---- roofline of the dominant kernel (the grouped MXFP4 gate/up GEMV)
    peaks, peak_kind = measured_peaks()
    kname = "gate/up"
    kern_ms, kern_bytes = 0.0, 0.0
    group_ms = {}
    for T in batches:
        for step_prof, n_act in zip(per_kernel[T], active_experts[T]):
            for name, ms in step_prof:
                group_ms.setdefault(name, []).append(ms)
                if name == kname:
                    kern_ms += ms
                    kern_bytes += n_act * d.expert_gate_up_bytes() + T * d.top_k * (d.latent + d.inter) * 2
    launches = sum(len(per_kernel[T]) for T in batches)
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9 if kern_ms > 0 else None
    path_used = layer.query("path_last")
    kernel_id = {1: "gateup_gemv_kernel", 4: "bs_stream_kernel_gateup"}[path_used]
    kernel_desc = {1: "gateup_gemv_kernel (CUDA-core grouped MXFP4 gate/up GEMV + SiTU-GLU)",
                   4: "bs_stream_kernel<GATEUP> (tcgen05 kind::mxf4: e2m1 weights as stored x six e2m1 "
                      "activation terms, UE8M0 scales in TMEM, SiTU-GLU + requantisation epilogue)"
                   }[path_used]
    # ncu's DRAM bytes per active expert (captured on a smaller case, traffic
    # grows with the experts touched) times this run's mean active experts
    per_expert = recorded_traffic(kernel_id, "k3-decode")
    mean_active = statistics.mean([n for T in batches for n in active_experts[T]])
    traffic = per_expert * mean_active if per_expert is not None else None
    roofline = {"bound": "hbm", "kernel": kernel_desc, "path": path_used,
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": (achieved / peaks["hbm_gbs"]) if achieved else None,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "traffic": traffic,
                "algorithmic_bytes_per_launch": kern_bytes / max(launches, 1)}
    # whole-layer HBM figure: all algorithmic bytes / forward time, per batch
    sweep = {}
    for T in batches:
        nact = statistics.mean(active_experts[T])
        alg = nact * d.expert_bytes() + d.dense_bytes() + T * d.hidden * 4
        fms = statistics.mean(fwd_ms[T])
        kms = {}
        for step_prof in per_kernel[T]:
            for name, ms in step_prof:
                kms.setdefault(name, []).append(ms)
        gu_ms = statistics.mean(kms.get(kname, [float("nan")]))
        gu_bytes = nact * d.expert_gate_up_bytes() + T * d.top_k * (d.latent + d.inter) * 2
        sweep[f"T={T}"] = {"forward_ms": fms, "tokens_per_s": T / (fms / 1e3), "active_experts": nact,
                           "algorithmic_GB": alg / 1e9, "layer_GB_per_s": alg / (fms / 1e3) / 1e9,
                           "gate_up_GB_per_s": gu_bytes / (gu_ms / 1e3) / 1e9,
                           "launches": launches_per_forward[T],
                           "kernel_ms": {k: statistics.mean(v) for k, v in kms.items()}}

    # ---- e2e: through the public C-ABI call with HOST buffers (pinned), copies timed
    t_leg = time.time()
    e2e = run_e2e(layer, d, batches, args, rank, dev, stream, l2_flush)
    clocks.mark("e2e", t_leg, time.time())
    t_leg = time.time()
    prefill = run_prefill(layer, d, prefill_T, rank, dev, stream, peaks) if prefill_T else None
    clocks.mark("prefill", t_leg, time.time())
    e2e_value = reduce_sum_over_ranks(e2e["tokens_per_s_rank"], world, dev)
    routed_step_ms = step_ms
    layer.close()
    torch.cuda.empty_cache()
    extra = {}
    if not args.no_extra and d.n_experts == K3.n_experts:
        t_leg = time.time()
        extra["shared_block"] = run_shared_block(w, args, rank, dev, stream, l2_flush, peaks, routed_step_ms)
        clocks.mark("shared_block", t_leg, time.time())
        t_leg = time.time()
        extra["two_bank"] = run_two_bank(w, d, args, rank, dev, stream, l2_flush, peaks, routed_step_ms)
        clocks.mark("two_bank", t_leg, time.time())
        torch.cuda.empty_cache()
        t_leg = time.time()
        extra["skew_4096"] = run_skew(w, rank, dev, stream, peaks)
        clocks.mark("skew_4096", t_leg, time.time())
        torch.cuda.empty_cache()
        if not args.no_stacked:
            t_leg = time.time()
            extra["stacked4"] = run_stacked4(args, rank, dev, l2_flush, peaks)
            clocks.mark("stacked4", t_leg, time.time())
    elif args.two_bank:  # a reduced-expert profiling case of the two-bank leg
        t_leg = time.time()
        extra["two_bank"] = run_two_bank(w, d, args, rank, dev, stream, l2_flush, peaks, routed_step_ms)
        clocks.mark("two_bank", t_leg, time.time())
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(d, w, args.cpu_sample)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 (e2m1 + e8m0) weights as stored; bf16 activations, carried to the block-scaled tensor "
                 "cores as six e2m1 terms (T <= 128) or two exact e4m3 terms (larger T); fp32 accumulate",
        "data": "synthetic (seeded generator: x~N(0,1) bf16, uniform MXFP4 bytes, e8m0 scales 118..124)",
        "config": {"workload": "K3 LatentMoE routed layer, decode batches T=1,8,64 per step (73 tokens)"
                   + ("" if d.n_experts == K3.n_experts else f" [reduced to {d.n_experts} experts: profiling case]"),
                   "hidden": d.hidden, "latent": d.latent, "experts": d.n_experts, "top_k": d.top_k,
                   "moe_intermediate": d.inter, "global_batch": tokens_per_step * world,
                   "l2": "flushed before every forward, outside the timed events (512 MB write, then a 256 MB read that leaves L2 clean)",
                   "timing": "CUDA events around each CUDA-graph replay of the C-ABI forward (graphs without per-kernel events); mean per batch size; kernel_ms from a separate replay of graphs captured with per-launch-group events",
                   "parallelism": f"replica x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "how": "k3moe_forward_host (pinned host x -> y, idx, w)"},
        "gpu_launches": sum(launches_per_forward[T] for T in batches) * args.steps,
        "decode_sweep": sweep,
        "wall_s_timed_region": t_wall,
    }
    if prefill is not None:
        out["prefill"] = prefill
    out.update(extra)
    if clk is not None:
        out["clocks"] = clk
        out["clocks_by_leg"] = clocks.window_summaries
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def run_prefill(layer, d, T, rank, dev, stream, peaks, reps: int = 5):
    """Prefill-size forward (T tokens, near-uniform routing): device time per
    forward with CUDA events, FLOP rate against the bf16 dense tensor peak.
    The forward touches every expert (15.8 GB of weights, far above L2), so
    no flush is needed between forwards."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    x = torch.from_numpy(synth.token_rows(d, 7000 + rank, T).view(np.int16)).to(dev)
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=dev)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=dev)
    wt = torch.empty((T, d.top_k), dtype=torch.float32, device=dev)
    k3moe.profile(layer.ctx, True)
    for _ in range(2):
        layer.forward(x, y, idx, wt, stream=stream)
    stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    kms = {}
    for i in range(reps):
        ev[i][0].record(stream)
        layer.forward(x, y, idx, wt, stream=stream)
        ev[i][1].record(stream)
        stream.synchronize()
        for name, ms in k3moe.profile_read(layer.ctx):
            kms.setdefault(name, []).append(ms)
    assert layer.status() == 0, k3moe.last_error(layer.ctx)
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    flop = d.flop_per_token() * T
    tflops = flop / (ms / 1e3) / 1e12
    peak = peaks.get("bf16_tflops") if isinstance(peaks, dict) else None
    return {"T": T, "ms_per_forward": ms, "tokens_per_s": T / (ms / 1e3), "algorithmic_tflop": flop / 1e12,
            "tflops": tflops, "bound": "tensor", "peak_bf16_tflops": peak,
            "frac": tflops / peak if peak else None,
            "peak_bf16_tflops_sustained": peaks.get("bf16_tflops_sustained") if isinstance(peaks, dict) else None,
            "path": layer.query("path_last"),
            "kernel_ms": {k: statistics.mean(v) for k, v in kms.items()},
            "how": f"CUDA events around each of {reps} forwards after 2 warm-up forwards; "
                   "FLOP = 2*(E*H + 2*L*H) + top_k*(2*2*I*L + 2*L*I) per token"}


def run_e2e(layer, d, batches, args, rank, dev, stream, l2_flush):
    """The public host-buffer call (k3moe_forward_host): pinned host x in,
    y / topk_idx / topk_w back to pinned host memory, copies inside the
    timed region; a fresh token batch every iteration and L2 flushed
    between iterations (outside the timed spans), as for `value`."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    k3moe.profile(layer.ctx, False)
    n = max(3, args.steps // 2)
    xs = {T: [torch.from_numpy(synth.token_rows(d, 9000 + 31 * rank + 7 * i + T, T).view(np.int16)).pin_memory()
              for i in range(n + 1)] for T in batches}
    ys = {T: torch.empty((T, d.hidden), dtype=torch.int16).pin_memory() for T in batches}
    ids = {T: torch.empty((T, d.top_k), dtype=torch.int32).pin_memory() for T in batches}
    ws = {T: torch.empty((T, d.top_k), dtype=torch.float32).pin_memory() for T in batches}
    for T in batches:
        k3moe.forward_host(layer.ctx, xs[T][n], T, ys[T], ids[T], ws[T], stream=stream)
    dt = 0.0
    for i in range(n):
        for T in batches:
            with torch.cuda.stream(stream):
                l2_flush()
            stream.synchronize()
            t0 = time.perf_counter()
            k3moe.forward_host(layer.ctx, xs[T][i], T, ys[T], ids[T], ws[T], stream=stream)
            dt += time.perf_counter() - t0
    dt /= n
    tok = sum(batches)
    h2d = sum(T * d.hidden * 2 for T in batches)
    d2h = sum(T * (d.hidden * 2 + d.top_k * 8) for T in batches)
    return {"tokens_per_s_rank": tok / dt, "h2d": h2d, "d2h": d2h}


# ============================================================================ further workloads
def _graph_decode(layer, d, T, reps, warmup, stream, l2_flush, seed0):
    """CUDA-graph replays of the C-ABI forward on fresh T-token batches, L2
    flushed before each (outside the events): (mean ms, mean active experts)."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    dev = stream.device
    xs = [torch.from_numpy(synth.token_rows(d, seed0 + 13 * i + T, T).view(np.int16)).to(dev)
          for i in range(warmup + reps)]
    x_in = torch.empty((T, d.hidden), dtype=torch.int16, device=dev)
    y = torch.empty((T, d.hidden), dtype=torch.int16, device=dev)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device=dev)
    wt = torch.empty((T, d.top_k), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        x_in.copy_(xs[0])
        layer.forward(x_in, y, idx, wt, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        layer.forward(x_in, y, idx, wt, stream=stream)
    ms, act = [], []
    for i in range(warmup + reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            l2_flush()
            x_in.copy_(xs[i])
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        if i >= warmup:
            ms.append(e0.elapsed_time(e1))
            a = np.empty(d.n_experts + 1, np.int32)
            k3moe.fetch(layer.ctx, "active", a)
            act.append(int(a[0]))
    assert layer.status() == 0, k3moe.last_error(layer.ctx)
    return statistics.mean(ms), statistics.mean(act)


def run_shared_block(w, args, rank, dev, stream, l2_flush, peaks, routed_step_ms):
    """The K3 MoE block with its two shared experts (bf16, 264 MB per layer,
    on a side stream beside the routed chain): the same decode step
    (T = 1, 8, 64) and the T = 8192 prefill."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    from mxfp4_routed_expert_k3_gb300.dims import K3_SHARED
    d = K3_SHARED
    ws = dict(w)
    ws.update(synth.shared_weights(d, seed=1))
    layer = k3moe.Layer(d, ws, max_tokens=PREFILL_T)
    try:
        per_T, step_ms, alg_bytes = {}, 0.0, 0.0
        for T in DECODE_BATCHES:
            ms, nact = _graph_decode(layer, d, T, max(5, args.steps // 2), args.warmup, stream, l2_flush, 11000)
            b = nact * d.expert_bytes() + d.dense_bytes() + d.shared_bytes() + T * d.hidden * 4
            per_T[f"T={T}"] = {"forward_ms": ms, "active_experts": nact, "algorithmic_GB": b / 1e9,
                               "GB_per_s": b / (ms / 1e3) / 1e9}
            step_ms += ms
            alg_bytes += b
        pf = run_prefill(layer, d, PREFILL_T, rank, dev, stream, peaks, reps=3)
    finally:
        layer.close()
    tok = sum(DECODE_BATCHES)
    return {"workload": "K3 MoE block: routed layer + 2 shared experts (intermediate 3072 each, bf16, on the "
                        "residual), decode batches T=1,8,64 per step",
            "tokens_per_s": tok / (step_ms / 1e3), "ms_per_step": step_ms,
            "shared_cost_ms_per_step": step_ms - routed_step_ms,
            "hbm_GB_per_s": alg_bytes / (step_ms / 1e3) / 1e9,
            "hbm_frac": alg_bytes / (step_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "decode": per_T, "prefill": pf}


def run_two_bank(w, d1, args, rank, dev, stream, l2_flush, peaks, routed_step_ms):
    """Two-bank graded experts: the first half of the experts MXFP4 (as in
    the main run), the second half 2-bit affine (2.5 bits per weight); the
    same decode step.  The banks' split of the sorted selections is found on
    the device."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    d = d1.with_(bank2_begin=d1.n_experts // 2)
    w2 = dict(w)
    for n in ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale"):
        w2[n] = np.ascontiguousarray(w[n][: d.bank2_begin])
    w2.update(synth.bank2_weights(d, seed=1))
    layer = k3moe.Layer(d, w2, max_tokens=max(DECODE_BATCHES))
    del w2
    try:
        per_T, step_ms, alg_bytes = {}, 0.0, 0.0
        for T in DECODE_BATCHES:
            ms, _ = _graph_decode(layer, d, T, max(5, args.steps // 2), args.warmup, stream, l2_flush, 13000)
            a = np.empty(d.n_experts + 1, np.int32)
            k3moe.fetch(layer.ctx, "active", a)
            ids = a[1:1 + a[0]]
            n1, n2 = int(np.sum(ids < d.bank2_begin)), int(np.sum(ids >= d.bank2_begin))
            b = n1 * d.expert_bytes() + n2 * d.expert_bytes_bank2() + d.dense_bytes() + T * d.hidden * 4
            per_T[f"T={T}"] = {"forward_ms": ms, "experts_bank1": n1, "experts_bank2": n2,
                               "algorithmic_GB": b / 1e9, "GB_per_s": b / (ms / 1e3) / 1e9}
            step_ms += ms
            alg_bytes += b
    finally:
        layer.close()
    tok = sum(DECODE_BATCHES)
    return {"workload": f"K3 routed layer, experts 0..{d.bank2_begin - 1} MXFP4 + {d.bank2_begin}.."
                        f"{d.n_experts - 1} 2-bit affine (second bank), decode batches T=1,8,64 per step",
            "tokens_per_s": tok / (step_ms / 1e3), "ms_per_step": step_ms,
            "vs_one_bank_time": step_ms / routed_step_ms,
            "hbm_GB_per_s": alg_bytes / (step_ms / 1e3) / 1e9, "decode": per_T}


def run_skew(w, rank, dev, stream, peaks, T: int = 4096, reps: int = 5):
    """Skewed routing (+2.0 correction bias on 32 hot experts, the first 32
    of a seeded permutation): every assignment lands on the hot set, about
    2,048 tokens per hot expert, 864 experts idle."""
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    from mxfp4_routed_expert_k3_gb300.dims import K3
    d = K3
    wk = dict(w)
    wk["router_bias"] = w["router_bias"].copy()
    wk["router_bias"][synth.hot_experts(d, 1, 32)] = np.float32(2.0)
    layer = k3moe.Layer(d, wk, max_tokens=T)
    try:
        r = run_prefill(layer, d, T, rank, dev, stream, peaks, reps=reps)
        counts = np.empty(d.n_experts, np.int32)
        k3moe.fetch(layer.ctx, "counts", counts)
    finally:
        layer.close()
    busy = counts[counts > 0]
    r.update({"workload": "K3 routed layer, T=4096, 32 hot experts (+2.0 bias)",
              "active_experts": int(busy.size), "tokens_per_hot_expert_max": int(busy.max()),
              "tokens_per_hot_expert_min": int(busy.min())})
    return r


def run_stacked4(args, rank, dev, l2_flush, peaks, n_layers: int = 4, T_pre: int = 32768):
    """Four stacked K3 routed layers (independent seeded weights, ~63 GB of
    MXFP4 experts resident), x_{l+1} = bf16(y_l / rms(y_l)) per token between
    layers: a T = 32768 prefill chain and a T = 1 decode chain, each captured
    in one CUDA graph and timed with events (decode: L2 flushed first)."""
    import torch
    from mxfp4_routed_expert_k3_gb300 import k3moe, synth
    from mxfp4_routed_expert_k3_gb300.dims import K3
    d = K3
    layers = []
    try:
        for l in range(n_layers):
            wl = synth.layer_weights(d, seed=4 + l)
            layers.append(k3moe.Layer(d, wl, max_tokens=T_pre, device=dev.index or 0))
            del wl
        s = torch.cuda.Stream(device=dev)

        def rescale(y):
            f = y.view(torch.bfloat16).float()
            return (f / torch.sqrt(torch.mean(f * f, dim=1, keepdim=True))).to(torch.bfloat16).view(torch.int16)

        def chain_graph(T, x0):
            xs = [torch.empty((T, d.hidden), dtype=torch.int16, device=dev) for _ in range(n_layers)]
            ys = [torch.empty((T, d.hidden), dtype=torch.int16, device=dev) for _ in range(n_layers)]
            ids = [torch.empty((T, d.top_k), dtype=torch.int32, device=dev) for _ in range(n_layers)]
            wts = [torch.empty((T, d.top_k), dtype=torch.float32, device=dev) for _ in range(n_layers)]

            def chain():
                for l, layer in enumerate(layers):
                    if l > 0:
                        xs[l].copy_(rescale(ys[l - 1]))
                    layer.forward(xs[l], ys[l], ids[l], wts[l], stream=s)

            xs[0].copy_(x0)
            with torch.cuda.stream(s):
                chain()
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                chain()
            return g, xs

        def timed(g, xs, pool, reps, warmup, flush):
            ms = []
            for i in range(warmup + reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(s):
                    if flush:
                        l2_flush()
                    xs[0].copy_(pool[i % len(pool)])
                    e0.record(s)
                    g.replay()
                    e1.record(s)
                s.synchronize()
                if i >= warmup:
                    ms.append(e0.elapsed_time(e1))
            for layer in layers:
                assert layer.status() == 0, k3moe.last_error(layer.ctx)
            return statistics.mean(ms)

        x_pre = torch.from_numpy(synth.token_rows(d, 12000 + rank, T_pre).view(np.int16)).to(dev)
        g_pre, xs_pre = chain_graph(T_pre, x_pre)
        pre_ms = timed(g_pre, xs_pre, [x_pre], reps=3, warmup=1, flush=False)
        del g_pre, xs_pre
        dec_pool = [torch.from_numpy(synth.token_rows(d, 12100 + 7 * i + rank, 1).view(np.int16)).to(dev)
                    for i in range(args.warmup + 10)]
        g_dec, xs_dec = chain_graph(1, dec_pool[0])
        dec_ms = timed(g_dec, xs_dec, dec_pool, reps=10, warmup=args.warmup, flush=True)
        act = []
        for layer in layers:
            a = np.empty(d.n_experts + 1, np.int32)
            k3moe.fetch(layer.ctx, "active", a)
            act.append(int(a[0]))
    finally:
        for layer in layers:
            layer.close()
        torch.cuda.empty_cache()
    flop = d.flop_per_token() * T_pre * n_layers
    dec_bytes = sum(a * d.expert_bytes() + d.dense_bytes() + 4 * d.hidden for a in act)
    peak = peaks.get("bf16_tflops")
    return {"workload": f"{n_layers} stacked K3 routed layers (seeds 4..{3 + n_layers}), per-token RMS rescale "
                        f"between layers, each chain one CUDA graph",
            "prefill": {"T": T_pre, "ms": pre_ms, "tokens_per_s": T_pre / (pre_ms / 1e3),
                        "tflops": flop / (pre_ms / 1e3) / 1e12, "frac_bf16_peak": flop / (pre_ms / 1e3) / 1e12 / peak,
                        "bound": "tensor"},
            "decode": {"T": 1, "ms": dec_ms, "tokens_per_s": 1 / (dec_ms / 1e3), "algorithmic_GB": dec_bytes / 1e9,
                       "GB_per_s": dec_bytes / (dec_ms / 1e3) / 1e9,
                       "hbm_frac": dec_bytes / (dec_ms / 1e3) / 1e9 / peaks["hbm_gbs"], "bound": "hbm",
                       "l2": "flushed before every replay"}}


# ============================================================================ oracle (CPU)
def cpu_baseline(d, w, n_tokens: int) -> dict:
    """The oracle, as it stands, on a bounded sample: n_tokens decode tokens
    through the whole layer on the host cores."""
    from mxfp4_routed_expert_k3_gb300 import synth
    from oracle import oracle as ora
    x = synth.token_rows(d, 7777, n_tokens)
    ora.forward(d, w, x[:1])  # load + page in
    t0 = time.perf_counter()
    ora.forward(d, w, x)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": ora.num_threads(), "kind": "oracle",
            "sample": f"{n_tokens} decode tokens of the K3 layer (full layer per token, fp64 oracle), "
                      f"{dt:.1f} s wall"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from mxfp4_routed_expert_k3_gb300 import synth
    from mxfp4_routed_expert_k3_gb300.dims import K3
    from oracle import oracle as ora
    d = K3
    w = synth.layer_weights(d, seed=1)
    # Bounded sample per step: one token per oracle thread by default.  The
    # oracle spreads tokens over its threads and a token's layer runs on one
    # thread, so a step costs about one token's time whatever its size up to
    # the thread count (about 13 s per step on 8-16 host cores).
    per_step = args.ref_tokens_per_step if args.ref_tokens_per_step > 0 else ora.num_threads()
    n_steps = args.warmup + args.steps
    xs = [synth.token_rows(d, 5000 + i, per_step) for i in range(n_steps)]
    for i in range(args.warmup):
        ora.forward(d, w, xs[i])
    times = []
    for i in range(args.warmup, args.warmup + args.steps):
        t0 = time.perf_counter()
        ora.forward(d, w, xs[i])
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    value = per_step / (ms / 1e3)
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (same generator and seed as the GPU arm)",
        "impl": "reference",
        "config": {"workload": "K3 LatentMoE routed layer, decode tokens (bounded sample per step)",
                   "tokens_per_step": per_step, "hidden": d.hidden, "latent": d.latent,
                   "experts": d.n_experts, "top_k": d.top_k, "moe_intermediate": d.inter},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ora.num_threads(), "kind": "oracle",
                         "sample": f"{per_step} decode tokens per step through the fp64 CPU oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=16, help="tokens in the oracle CPU baseline sample")
    ap.add_argument("--ref-tokens-per-step", type=int, default=0,
                    help="tokens per step of the reference arm (0: one per oracle thread)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the T=8192 prefill measurement")
    ap.add_argument("--prefill-tokens", type=int, default=PREFILL_T,
                    help="tokens of the prefill measurement (default 8192; with --experts E, 8192*E/896 keeps "
                         "the tokens per expert of the full layer, for small profiling captures)")
    ap.add_argument("--path", type=int, default=0, choices=[0, 1, 4],
                    help="kernel path (0 = the library's choice by token count; see k3moe_config.force_path)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the shared-expert block, skewed-routing and stacked-layer measurements")
    ap.add_argument("--no-stacked", action="store_true", help="skip the four-stacked-layer measurement")
    ap.add_argument("--two-bank", action="store_true",
                    help="with --experts below 896: run the two-bank leg at that expert count (profiling case)")
    ap.add_argument("--experts", type=int, default=896,
                    help="experts of the K3-dim layer (default 896; fewer only for small profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_info()
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
