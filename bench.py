#!/usr/bin/env python
"""Benchmark of the fused attention hot path on GB300.

One step = the whole path once: fa_fwd (O, LSE) then fa_bwd (dQ, dK, dV) with the
variant the library picks for the shape, on synthetic inputs drawn by
``tiled_attention_tmem_gb300.inputs`` (i.i.d. normal, bf16).  Throughput counts
nominal FLOPs: 4*B*H*N^2*d for the forward, 2.5x that for the backward, both
halved under the causal mask.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Rank 0 prints one JSON line.  With N > 1 (launched by torch.distributed.run)
every rank runs its own replica of the workload on its own GPU (the path has no
cross-GPU exchange); the value is the total FLOPs of all ranks over the slowest
rank's time.  ``--impl reference`` times the CPU fp64 oracle on a bounded sample
of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS, bf16 d=128, and % of GB300 dense BF16 tensor peak"
DEFAULT_WORKLOAD = "b4_h16_n2048_d128_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch of the dominant kernel, read from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum).  Keyed by the workload and the
# hash of the kernel sources it was taken on; any source change voids it.
NCU_TRAFFIC = {
    ("b4_h16_n2048_d128_causal", "bwd_kv5", "bdd7365a73e89c76"): 310.8e6,
    ("b4_h16_n2048_d128_causal", "fwd", "bdd7365a73e89c76"): 156.6e6,
    ("b4_h16_n2048_d128_causal", "bwd_kv7", "bdd7365a73e89c76"): 170.7e6,
    ("b4_h16_n2048_d128_causal", "bwd_q7", "bdd7365a73e89c76"): 154.6e6,
    ("b2_h16_n8192_d128_kshift3", "fwd", "bdd7365a73e89c76"): 377.4e6,
    ("b2_h16_n8192_d128_kshift3", "bwd_kv5", "bdd7365a73e89c76"): 943.9e6,
    ("b2_h8_n4096_d256_causal_sigma0.5", "bwd_kv7", "bdd7365a73e89c76"): 175.8e6,
    ("b2_h8_n4096_d256_causal_sigma0.5", "bwd_q7", "bdd7365a73e89c76"): 197.8e6,
    ("b2_h8_n4096_d256_causal_sigma0.5", "fwd", "bdd7365a73e89c76"): 159.5e6,
    ("b2_h8_n4096_d384_causal_sigma0.5", "bwd_kv7", "bdd7365a73e89c76"): 280.0e6,
    ("b1_h1_n16384_d128_causal", "bwd_kv5", "bdd7365a73e89c76"): 46.7e6,
    ("b1_h1_n8192_d256_causal_sigma0.5", "bwd_q7", "bdd7365a73e89c76"): 22.3e6,
    ("b1_h1_n8192_d256_causal_sigma0.5", "bwd_kv7", "bdd7365a73e89c76"): 29.0e6,
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--variant", choices=["auto", "5", "7"], default="auto")
    ap.add_argument("--splits", default="auto",
                    help="forward key parts per query block: 'auto' (the library's cost model) or a count")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--variant-table", action="store_true",
                    help="time the 5-GEMM and 7-GEMM backward over a grid of shapes (one JSON line per point)")
    ap.add_argument("--split-table", action="store_true",
                    help="time the backward with the dK/dV query range forced to 1..8 parts (few heads)")
    ap.add_argument("--key-split-table", action="store_true",
                    help="time the 7-GEMM backward with the dQ kernel's key range forced to 1..12 parts (few heads)")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the timed pass of K steps until this long has elapsed (median pass reported)")
    return ap.parse_args()


def kernel_source_hash() -> str:
    """Hash of the CUDA sources with // comments and blank lines removed, so that a
    change to comments alone keeps the recorded ncu traffic valid."""
    d = os.path.join(ROOT, "tiled_attention_tmem_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            code = []
            for line in fh:
                s = line.split("//", 1)[0].rstrip()
                if s:
                    code.append(s)
        h.update(f.encode() + "\n".join(code).encode())
    return h.hexdigest()[:16]


def aggregate_throughput(local_seconds: float, flops_per_step: float, steps: int, device=None) -> tuple[float, float]:
    """Whole-job TFLOP/s of a replicated run: every rank ran `steps` steps of the same
    workload; the job's time is the slowest rank's.  Returns (TFLOP/s, max seconds)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    tmax = float(t.item())
    return flops_per_step * steps * world / tmax / 1e12, tmax


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines: list[str] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
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
        time.sleep(0.25)
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
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ exp-unit probe


def measure_ex2(b, dev, stream, iters: int = 4096, repeats: int = 5) -> dict:
    """ex2.approx evaluations per second of the library's probe kernel on this GPU:
    8 CTAs of 256 threads per SM, each thread 8 independent chains of `iters`
    evaluations; best of `repeats` launches timed with CUDA events on `stream`."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = 8 * sms
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    best = None
    count = 0
    for r in range(repeats + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st, count = b.fa_ex2_probe(sink.data_ptr(), blocks, iters, stream.cuda_stream)
        e1.record(stream)
        if st != b.FA_OK:
            raise b.FaError(st, "fa_ex2_probe")
        torch.cuda.synchronize()
        if r >= 2:  # two untimed launches first
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
    return {"ex2_per_s": count / (best / 1e3),
            "how": f"fa_ex2_probe: {count} ex2.approx.ftz.f32 in {blocks} CTAs x 256 threads, "
                   f"best of {repeats} launches, {best:.3f} ms"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or '' if neither says."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


# --------------------------------------------------------------- oracle timing


def time_oracle(w, seconds: float, max_heads: int | None = None):
    """Times the fp64 CPU oracle (forward + backward) on whole heads of the workload."""
    import numpy as np

    import oracle
    from tiled_attention_tmem_gb300 import inputs as I
    x = I.make_inputs(1, 1, w.N, w.d, seed=w.seed, sigma=w.sigma, k_shift=w.k_shift)
    q, k, v, do = x.as_f64()
    heads = 0
    t0 = time.perf_counter()
    while True:
        oracle.forward(q, k, v, w.softmax_scale, w.causal)
        oracle.backward(q, k, v, do, w.softmax_scale, w.causal)
        heads += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_heads is not None and heads >= max_heads):
            break
    per_head = (w.fwd_flops + w.bwd_flops) / (w.B * w.H)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": per_head * heads / el / 1e12, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": f"{heads} whole heads of {w.name} (a head is 1 of its B*H={w.B * w.H}), fp64 numpy with "
                      f"multithreaded BLAS matmuls, forward + backward, {el:.1f} s",
            "seconds": el}


# -------------------------------------------------------------------- arms


def run_reference(args, rank, world):
    from tiled_attention_tmem_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    if rank != 0:
        return
    per_head = (w.fwd_flops + w.bwd_flops) / (w.B * w.H)
    # Each step is one whole head: a bounded sample of the workload.
    for _ in range(args.warmup):
        time_oracle(w, 0.0, max_heads=1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(w, 0.0, max_heads=1)
    el = time.perf_counter() - t0
    value = per_head * args.steps / el / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "step_sample": "one whole head (b=0, h=0) per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                         "kind": "oracle",
                         "sample": "one whole head per step, fp64 numpy oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    from tiled_attention_tmem_gb300 import api, binding as b, build, inputs as I

    build.build_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = I.WORKLOADS[args.workload]
    variant = {"auto": b.FA_BWD_AUTO, "5": b.FA_BWD_5GEMM, "7": b.FA_BWD_7GEMM}[args.variant]
    chosen = variant if variant != b.FA_BWD_AUTO else b.fa_bwd_choose(w.B, w.H, w.N, w.d, w.causal)

    x = I.workload_inputs(w)
    host = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
            for a in (x.q, x.k, x.v, x.do)]
    q, k, v, do = (t.to(dev) for t in host)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    ws = torch.empty(b.fa_bwd_workspace_size(w.B, w.H, w.N, w.d, chosen), dtype=torch.uint8, device=dev)
    splits = (b.fa_fwd_choose_splits(w.B, w.H, w.N, w.d, w.causal) if args.splits == "auto"
              else int(args.splits))
    split_ws = torch.empty(max(1, b.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.d, splits)),
                           dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > 129 MB L2
    scale = w.softmax_scale
    stream = torch.cuda.current_stream()

    def step():
        api.attention_forward(q, k, v, scale, w.causal, out=o, lse=lse, splits=splits, workspace=split_ws)
        api.attention_backward(q, k, v, o, do, lse, scale, w.causal, variant=chosen, workspace=ws,
                               grads=grads)

    for _ in range(max(args.warmup, 3)):
        step()
    api.check_device_error()

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)

    def timed_pass(profiled: bool):
        """K steps, L2 flushed between them (outside the events); per-step device times in ms.
        With profiled=True the library also records events around each of its kernels."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        if profiled:
            b.fa_profile_start()
        for i in range(args.steps):
            flush.fill_(float(i))  # evict L2 between timed steps (outside the events)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        prof_ = b.fa_profile_stop() if profiled else None
        if world > 1:
            dist.barrier()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], prof_

    # Headline: passes of exactly K steps, nothing but the steps between the per-step
    # events, repeated until about a second has gone by so that the clock sampler sees
    # the GPU under load many times; the pass with the median time is reported.  A
    # second, instrumented pass of the same steps gives the per-kernel times (the
    # library's per-kernel events add about 16 us per step, so they stay out of the
    # headline).
    t_first = time.perf_counter()
    passes = [timed_pass(profiled=False)[0]]
    more = min(999, max(0, math.ceil(args.min_seconds / max(time.perf_counter() - t_first, 1e-3)) - 1))
    if world > 1:  # every rank runs the same number of passes (each pass has barriers)
        t_more = torch.tensor([more], dtype=torch.int64, device=dev)
        dist.all_reduce(t_more, op=dist.ReduceOp.MAX)
        more = int(t_more.item())
    for _ in range(more):
        passes.append(timed_pass(profiled=False)[0])
    passes.sort(key=sum)
    times_ms = passes[len(passes) // 2]
    ex2_probe = measure_ex2(b, dev, stream)
    clocks = sampler.stop()
    api.check_device_error()
    # The library creates its profiling events on first use: one untimed profiled pass
    # fills its event pool so that no event is created inside the instrumented pass.
    b.fa_profile_start()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    b.fa_profile_stop()
    prof_times_ms, prof = timed_pass(profiled=True)
    api.check_device_error()
    flops_step = w.fwd_flops + w.bwd_flops
    value, total_s = aggregate_throughput(sum(times_ms) / 1e3, flops_step, args.steps, dev)
    pass_values = [flops_step * args.steps / (sum(t_) / 1e3) / 1e12 for t_ in passes]
    launches = args.steps * (b.fa_fwd_splitkv_launches(w.B, w.H, w.N, w.d, splits)
                             + b.fa_bwd_launches(w.B, w.H, w.N, w.d, chosen, w.causal))
    assert sum(n for n, _ in prof.values()) == launches, "launch count mismatch"

    # Per-kernel timing from the library's own events (same stream as the kernels).
    n_bh_flops = {
        "fwd": w.fwd_flops,
        "bwd_kv5": w.bwd_flops,           # S, dP, dV, dK, dQ: all five GEMMs
        "bwd_kv7": w.bwd_flops * 4 / 5,   # S, dP, dV, dK
        "bwd_q7": w.bwd_flops * 3 / 5,    # S, dP, dQ
    }
    kernels = {}
    for name, (n, ms) in prof.items():
        if n:
            kernels[name] = {"launches": n, "ms_avg": ms / n, "share": None}
    tot_ms = sum(v_["ms_avg"] * v_["launches"] for v_ in kernels.values())
    for v_ in kernels.values():
        v_["share"] = v_["ms_avg"] * v_["launches"] / tot_ms if tot_ms else None
    dominant = max(kernels, key=lambda n_: kernels[n_]["ms_avg"] * kernels[n_]["launches"])
    peaks, peak_src = load_peaks()
    roof = None
    if dominant in n_bh_flops:
        ach = n_bh_flops[dominant] / (kernels[dominant]["ms_avg"] / 1e3) / 1e12
        peak = float(peaks["bf16_tflops"])
        tr = NCU_TRAFFIC.get((w.name, dominant, kernel_source_hash()))
        roof = {"bound": "tensor", "kernel": dominant, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak, "traffic": tr, "traffic_unit": "bytes per launch (ncu dram read + write)",
                "peak_source": f"bf16_tflops (burst) of {peak_src} peaks",
                "frac_of_sustained": ach / float(peaks["bf16_tflops_sustained"])}
    fwd_ms = sum(kernels[n_]["ms_avg"] for n_ in ("fwd", "fwd_merge") if n_ in kernels)
    fwd_tf = w.fwd_flops / (fwd_ms / 1e3) / 1e12 if fwd_ms else None
    bwd_ms = sum(kernels[n_]["ms_avg"] for n_ in ("bwd_pre", "bwd_kv5", "bwd_conv", "bwd_kv7", "bwd_q7",
                                                  "bwd_kvsum", "bwd_qsum")
                 if n_ in kernels)
    bwd_tf = w.bwd_flops / (bwd_ms / 1e3) / 1e12 if bwd_ms else None

    # The exp-unit bound of the method (one ex2 per score in the forward and the
    # 5-GEMM backward, two in the 7-GEMM backward): nominal FLOPs per exp x the ex2
    # rate, measured in this run by the library's probe (fa_ex2_probe: ex2.approx
    # evaluations over CUDA-event time on this stream), per SM per clock at the
    # median SM clock sampled during the timed passes.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk = ((clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))) * 1e6
    ex2_rate = ex2_probe["ex2_per_s"]
    ex2_per_sm_clk = ex2_rate / sms / clk
    exps_bwd = 1 if chosen == b.FA_BWD_5GEMM else 2
    exp_fwd_tf = 4 * w.d * ex2_rate / 1e12
    exp_bwd_tf = 10 * w.d * ex2_rate / exps_bwd / 1e12
    exp_bound = {"source": "measured", "ex2_per_s": ex2_rate, "ex2_per_sm_clk": ex2_per_sm_clk,
                 "probe": ex2_probe["how"], "fwd_tflops": exp_fwd_tf, "bwd_tflops": exp_bwd_tf,
                 "fwd_frac": fwd_tf / exp_fwd_tf if fwd_tf else None,
                 "bwd_frac": bwd_tf / exp_bwd_tf if bwd_tf else None}

    # The instruction metric of the Metal FlashAttention benchmark quoted in "Potential
    # algorithmic improvements for backward pass" (head-dim sweep): per visible score,
    # 2d + 5 instructions in the forward, 3d + 5 in a dQ kernel (S, dP, dQ) and 4d + 5 in a
    # dK/dV kernel (S, dP, dV, dK), i.e. d multiply-adds per GEMM plus five softmax
    # instructions; the 5-GEMM kernel runs all five GEMMs (5d + 5).  Giga-instructions/s per
    # kernel from its measured time, scores halved under the causal mask like the FLOPs.
    scores = float(w.B * w.H) * w.N * w.N * (0.5 if w.causal else 1.0)
    per_score = {"fwd": 2 * w.d + 5, "bwd_kv5": 5 * w.d + 5, "bwd_kv7": 4 * w.d + 5, "bwd_q7": 3 * w.d + 5}
    instr_metric = {name_: per_score[name_] * scores / (kernels[name_]["ms_avg"] / 1e3) / 1e9
                    for name_ in per_score if name_ in kernels}
    instr_metric["unit"] = "GINSTRS (per-score instruction counts of the Metal FlashAttention benchmark)"

    # The HBM-bound helper kernels against the measured copy bandwidth:
    # algorithmic bytes per launch / average launch time.
    npad = (w.N + 127) // 128 * 128
    dk_ = 64 if w.d <= 64 else (128 if w.d <= 128 else 256)  # kernel head dim (96 -> 128)
    bh = w.B * w.H
    hbm_bytes = {
        # O, dO and LSE read; log2-domain LSE and D written; 5-GEMM: fp32 dQ accumulator zeroed
        "bwd_pre": 2 * bh * w.N * w.d * 2 + 4 * bh * w.N + 8 * bh * npad
        + (4 * bh * npad * dk_ if chosen == b.FA_BWD_5GEMM else 0),
        # fp32 dQ accumulator read, bf16 dQ written
        "bwd_conv": 4 * bh * w.N * dk_ + 2 * bh * w.N * w.d,
        # split-KV merge: fp32 parts and their log-sum-exps read, bf16 O and LSE written
        "fwd_merge": 4 * splits * bh * w.N * (w.d + 1) + 2 * bh * w.N * w.d + 4 * bh * w.N,
        # backward splits: fp32 partial dK and dV (dQ) of every part read, bf16 written
        "bwd_kvsum": 2 * (4 * b.fa_bwd_query_parts(w.B, w.H, w.N, w.d, w.causal, chosen) + 2) * bh * w.N * w.d,
        "bwd_qsum": (4 * b.fa_bwd_key_parts(w.B, w.H, w.N, w.d, w.causal, chosen) + 2) * bh * w.N * w.d,
    }
    hbm = {}
    for name_, bytes_ in hbm_bytes.items():
        if name_ in kernels:
            gbs = bytes_ / (kernels[name_]["ms_avg"] / 1e3) / 1e9
            hbm[name_] = {"bytes": bytes_, "GB/s": gbs, "frac": gbs / float(peaks["hbm_gbs"])}

    # End to end through the public API: every step copies its Q, K, V, dO from
    # pinned host memory to the device and its O, LSE, dQ, dK, dV back to pinned
    # host memory.  Steps are pipelined over two sets of device buffers and three
    # streams (copy in, compute, copy out), so a step's copies overlap its
    # neighbours' compute; the timed region runs from the first copy in to the
    # last copy out.
    out_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, *grads)]
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    nbuf = 2
    dev_in = [[torch.empty_like(t_) for t_ in (q, k, v, do)] for _ in range(nbuf)]
    dev_out = [(torch.empty_like(o), torch.empty_like(lse)) + tuple(torch.empty_like(g_) for g_ in grads)
               for _ in range(nbuf)]
    # Copy streams per direction (more than one measured no faster: the copies are
    # bound by the host link).
    n_cs = 1
    s_in = [torch.cuda.Stream() for _ in range(n_cs)]
    s_out = [torch.cuda.Stream() for _ in range(n_cs)]
    s_cmp = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(nbuf)]

    def e2e_run(n_steps):
        for i in range(n_steps):
            bi = i % nbuf
            for c in range(n_cs):
                if i >= nbuf:
                    s_in[c].wait_event(ev_cmp[bi])  # step i-2 has finished reading these inputs
                with torch.cuda.stream(s_in[c]):
                    for j_, (hsrc, ddst) in enumerate(zip(host, dev_in[bi])):
                        if j_ % n_cs == c:
                            ddst.copy_(hsrc, non_blocking=True)
                    ev_in[bi][c].record(s_in[c])
                s_cmp.wait_event(ev_in[bi][c])
                if i >= nbuf:
                    s_cmp.wait_event(ev_out[bi][c])  # step i-2's outputs have been copied out
            qq, kk, vv, dd_ = dev_in[bi]
            oo, ll, gq, gk, gv = dev_out[bi]
            api.attention_forward(qq, kk, vv, scale, w.causal, out=oo, lse=ll, stream=s_cmp.cuda_stream,
                                  splits=splits, workspace=split_ws)
            api.attention_backward(qq, kk, vv, oo, dd_, ll, scale, w.causal, variant=chosen, workspace=ws,
                                   grads=(gq, gk, gv), stream=s_cmp.cuda_stream)
            ev_cmp[bi].record(s_cmp)
            for c in range(n_cs):
                s_out[c].wait_event(ev_cmp[bi])
                with torch.cuda.stream(s_out[c]):
                    for j_, (hdst, dsrc) in enumerate(zip(out_host, dev_out[bi])):
                        if j_ % n_cs == c:
                            hdst.copy_(dsrc, non_blocking=True)
                    ev_out[bi][c].record(s_out[c])

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_.record(s_in[0])
    for c in range(1, n_cs):
        s_in[c].wait_event(s_)
    e2e_run(e2e_steps)
    for st_ in s_in[1:] + s_out + [s_cmp]:
        s_in[0].wait_stream(st_)
    e_.record(s_in[0])
    torch.cuda.synchronize()
    e2e_val, _ = aggregate_throughput(s_.elapsed_time(e_) / 1e3, flops_step, e2e_steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in out_host)
    api.check_device_error()

    cpu = None
    if rank == 0 and world == 1:
        cpu = time_oracle(w, args.cpu_seconds)
        cpu.pop("seconds", None)

    if rank == 0:
        frac = value / world / float(peaks["bf16_tflops"])
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                       "scale": scale, "bwd_variant": f"{chosen}-GEMM" + (" (auto)" if variant == 0 else ""),
                       "fwd_splits": splits,
                       "l2": "flushed (256 MiB write) between timed steps, outside the timed events",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "frac_of_peak": frac, "peak_tflops": float(peaks["bf16_tflops"]),
            "roofline": roof, "exp_bound": exp_bound, "instr_metric": instr_metric, "hbm_kernels": hbm,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "pipelining": "copy in / compute / copy out on three streams, two device buffer sets"},
            "gpu_launches": launches, "kernels": kernels,
            "kernel_timing": ("per-kernel events in a second pass of the same steps "
                              f"({sum(prof_times_ms) / args.steps:.4f} ms per step with them)"),
            "clocks": clocks,
            "timed_passes": {"count": len(passes), "steps_each": args.steps, "reported": "median pass",
                             "min_tflops": min(pass_values), "max_tflops": max(pass_values)},
        }
        print(json.dumps(line), flush=True)


def variant_grid():
    """(d, causal, B*H, N) points of the 5-GEMM / 7-GEMM comparison: N from 512 to
    16384, one to 512 heads, capped at B*H*N^2 <= 2^32 so that a point stays short."""
    pts = []
    for d in (64, 96, 128):
        for causal in (False, True):
            for n in (512, 1024, 2048, 4096, 8192, 16384):
                for bh in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
                    if bh * n * n <= 1 << 32:
                        pts.append((d, causal, bh, n))
    return pts


def run_variant_table(args):
    """Times fa_bwd with the 5-GEMM and the 7-GEMM form at every point of
    variant_grid() (CUDA events on the launching stream, L2 flushed between calls,
    best of --steps calls after --warmup) and prints one JSON line per point with
    both times and the faster form: the measurements behind fa_bwd_choose."""
    import torch

    from tiled_attention_tmem_gb300 import api, binding as b, build

    build.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    for d, causal, bh, n in variant_grid():
        gen.manual_seed(1000003 * d + 1009 * n + bh + (7 if causal else 0))
        shape = (1, bh, n, d)
        q, k, v, do = (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                       for _ in range(4))
        scale = d ** -0.5
        o, lse = api.attention_forward(q, k, v, scale, causal)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        ws = torch.empty(b.fa_bwd_workspace_size(1, bh, n, d, b.FA_BWD_AUTO), dtype=torch.uint8, device=dev)
        ms = {}
        for variant in (b.FA_BWD_5GEMM, b.FA_BWD_7GEMM):
            best = None
            for i in range(args.warmup + args.steps):
                flush.fill_(float(i))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant, workspace=ws,
                                       grads=grads)
                e1.record(stream)
                torch.cuda.synchronize()
                if i >= args.warmup:
                    t = e0.elapsed_time(e1)
                    best = t if best is None else min(best, t)
            ms[variant] = best
        api.check_device_error()
        flops = 10.0 * bh * n * n * d * (0.5 if causal else 1.0)
        print(json.dumps({"d": d, "causal": causal, "BH": bh, "N": n,
                          "ms5": ms[5], "ms7": ms[7], "tflops5": flops / ms[5] / 1e9, "tflops7": flops / ms[7] / 1e9,
                          "faster": 5 if ms[5] <= ms[7] else 7,
                          "auto": b.fa_bwd_choose(1, bh, n, d, int(causal))}), flush=True)


def split_grid():
    """(B*H, N, d, causal, variant) points of the query-split sweep: few heads (the
    dK/dV kernel's items below two per SM), N = 2048 to 16384, both masks."""
    pts = []
    for d in (64, 128):
        for causal in (True, False):
            for n in (2048, 4096, 8192, 16384):
                for bh in (1, 2, 4, 8, 16):
                    if bh * (n // 128) < 304:
                        pts.append((bh, n, d, causal, 5))
    pts += [(1, 8192, 256, True, 7), (2, 8192, 256, True, 7), (1, 16384, 256, True, 7), (4, 4096, 256, True, 7),
            (1, 8192, 384, True, 7), (2, 4096, 384, True, 7), (1, 8192, 192, True, 7), (1, 8192, 256, False, 7)]
    return pts


def run_split_table(args):
    """Times fa_bwd at every point of split_grid() with the dK/dV kernel's query range
    forced to 1, 2, 3, 4, 6 and 8 parts (fa_bwd_force_query_parts; CUDA events, L2
    flushed, best of --steps calls after --warmup) and prints one JSON line per point
    with the times and the part count the library's rule picks: the measurements the
    rule was fitted to."""
    import torch

    from tiled_attention_tmem_gb300 import api, binding as b, build

    build.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    for bh, n, d, causal, variant in split_grid():
        gen.manual_seed(7919 * d + 31 * n + bh + (3 if causal else 0))
        q, k, v, do = (torch.randn((1, bh, n, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                       for _ in range(4))
        scale = d ** -0.5
        o, lse = api.attention_forward(q, k, v, scale, causal)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        auto = b.fa_bwd_query_parts(1, bh, n, d, int(causal), variant)
        ms = {}
        for parts in (1, 2, 3, 4, 6, 8):
            b.fa_bwd_force_query_parts(parts)
            try:
                ws = torch.empty(b.fa_bwd_workspace_size(1, bh, n, d, variant), dtype=torch.uint8, device=dev)
                best = None
                for i in range(args.warmup + args.steps):
                    flush.fill_(float(i))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=variant, workspace=ws,
                                           grads=grads)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if i >= args.warmup:
                        t = e0.elapsed_time(e1)
                        best = t if best is None else min(best, t)
            finally:
                b.fa_bwd_force_query_parts(0)
            ms[parts] = best
        api.check_device_error()
        print(json.dumps({"BH": bh, "N": n, "d": d, "causal": causal, "variant": variant, "ms": ms,
                          "fastest": min(ms, key=ms.get), "rule": auto}), flush=True)


def key_split_grid():
    """(B*H, N, d, causal) points of the key-split sweep: the 7-GEMM dQ kernel's work
    items (query tiles x dQ column parts x heads) below two per SM, N = 2048 to 16384,
    d = 64 to 384, both masks."""
    pts = []
    for d in (64, 128, 192, 256, 384):
        dqs = 2 if d == 384 else 1
        for causal in (True, False):
            for n in (2048, 4096, 8192, 16384):
                for bh in (1, 2, 4, 8, 16):
                    if bh * (n // 128) * dqs < 304 and not (d == 384 and n == 16384):
                        pts.append((bh, n, d, causal))
    return pts


def run_key_split_table(args):
    """Times the 7-GEMM fa_bwd at every point of key_split_grid() with the dQ kernel's
    key range forced to 1, 2, 3, 4, 6, 8 and 12 parts (fa_bwd_force_key_parts; the
    query split left to the library; CUDA events, L2 flushed, best of --steps calls
    after --warmup) and prints one JSON line per point with the times and the part
    count the library's rule picks."""
    import torch

    from tiled_attention_tmem_gb300 import api, binding as b, build

    build.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    for bh, n, d, causal in key_split_grid():
        gen.manual_seed(7907 * d + 29 * n + bh + (5 if causal else 0))
        q, k, v, do = (torch.randn((1, bh, n, d), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
                       for _ in range(4))
        scale = d ** -0.5
        o, lse = api.attention_forward(q, k, v, scale, causal)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        auto = b.fa_bwd_key_parts(1, bh, n, d, int(causal), b.FA_BWD_7GEMM)
        ms = {}
        for parts in (1, 2, 3, 4, 6, 8, 12):
            b.fa_bwd_force_key_parts(parts)
            try:
                ws = torch.empty(b.fa_bwd_workspace_size(1, bh, n, d, b.FA_BWD_7GEMM), dtype=torch.uint8,
                                 device=dev)
                best = None
                for i in range(args.warmup + args.steps):
                    flush.fill_(float(i))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    api.attention_backward(q, k, v, o, do, lse, scale, causal, variant=b.FA_BWD_7GEMM,
                                           workspace=ws, grads=grads)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if i >= args.warmup:
                        t = e0.elapsed_time(e1)
                        best = t if best is None else min(best, t)
            finally:
                b.fa_bwd_force_key_parts(0)
            ms[parts] = best
        api.check_device_error()
        print(json.dumps({"BH": bh, "N": n, "d": d, "causal": causal, "ms": ms,
                          "fastest": min(ms, key=ms.get), "rule": auto}), flush=True)


def main():
    args = parse_args()
    if args.key_split_table:
        run_key_split_table(args)
        return
    if args.variant_table:
        run_variant_table(args)
        return
    if args.split_table:
        run_split_table(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, rank, world)
        if world > 1:
            dist.destroy_process_group()
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
