#!/usr/bin/env python
"""Benchmark of the fused LongFlow decode step (attention + LongFlowScore +
eviction) on GB300.

Default workload: the Qwen3-8B Fig. 1 shape of "LongFlow: Efficient KV Cache
Compression for Reasoning Models" (batch 128, 32 query / 8 KV heads, head dim
128, 3200 cache slots, W = 32), with synthetic seeded bf16 data.

A step is one call of lf_decode_step over the whole batch: slot write, mask
ageing, attention, score and argmin for every (b, kvh) unit. The step's
write_slot is the previous step's next_slot (every-step eviction), kept on the
device. Inputs are resident in HBM before timing starts; the K/V caches
(1.68 GB) are far larger than the 129 MB L2, so no flush is needed.

Output: one JSON line on rank 0 (see the keys at the end of main()).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores
Under torchrun each rank runs its own batch of sequences (weak scaling, no
collective on the data path); the time reported is the max over ranks.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from decode_kv_cache_step_gb300.workloads import (  # noqa: E402
    WORKLOADS, algorithmic_bytes, initial_state, live_lengths, step_inputs)

METRIC = "decode steps/s and achieved HBM GB/s (% of GB300 peak) for fused attn+score+evict"
DEFAULT_WORKLOAD = "qwen3_8b_b128_s3200"
FALLBACK_HBM_GBS = 6800.0
PROFILE_WORKLOAD = "qwen3_8b_b128_s3200"   # the workload the committed DRAM counters cover
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", f"lf_decode_step_kernel.{PROFILE_WORKLOAD}.md")
KERNEL_SOURCES = ["lf_step_kernel.cuh", "lf_decode_step.cu", "lf_decode_step_cluster.cu",
                  "lf_ptx.cuh", "lf_kernels.h"]


def kernel_source_hash() -> str:
    """Hash of the kernel's sources with comments and blank lines removed, so
    that the committed ncu counters stay tied to the code, not its comments."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "decode_kv_cache_step_gb300", "csrc", name)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(text.encode())
    return h.hexdigest()[:16]


def committed_traffic():
    """dram read+write bytes per launch of the decode-step kernel from the committed ncu
    summary, or None if absent or taken on another version of the kernel."""
    try:
        with open(PROFILE_SUMMARY) as fh:
            text = fh.read()
    except OSError:
        return None
    src, traffic = None, None
    for line in text.splitlines():
        if line.startswith("source_sha:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    if src != kernel_source_hash():
        return None
    return traffic


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return json.load(fh), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms), "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.monotonic(), parts))

    def mark(self):
        return time.monotonic()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [r for t, r in self.rows if t0 - 0.06 <= t <= t1 + 0.06] or [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def bf16_dev(a, device):
    import torch
    return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def run_oracle_steps(wl, state, max_seconds: float, max_steps: int, units=None, nthreads=0):
    """Times oracle steps (the CPU baseline); returns (steps, seconds, threads,
    per-step seconds). nthreads = 0 uses every OpenMP thread."""
    import oracle
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)
    done, t_total, times = 0, 0.0, []
    while done < max_steps and (t_total < max_seconds or done == 0):
        inp = step_inputs(wl, 1000 + done)
        t0 = time.perf_counter()
        res = oracle.decode_step(inp["q"], state["k_cache"], state["v_cache"], state["mask"],
                                 inp["new_k"], inp["new_v"], ws, wl.W, wl.scale, units=units,
                                 nthreads=nthreads)
        times.append(time.perf_counter() - t0)
        t_total += times[-1]
        ws = res["next_slot"].copy()
        if units is not None:
            ws[ws < -1] = -1
        done += 1
    return done, t_total, (nthreads if nthreads > 0 else oracle.max_threads()), times


def bench_reference(args, wl):
    """The fp64 CPU oracle on the host cores. Each timed step is a whole step
    (every (b, kvh) unit) when the K steps fit in --reference-seconds at the
    warm-up steps' rate; otherwise each step runs the same sample of units,
    sized to fit, and the line says so."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    st = initial_state(wl)
    k, v, mask = st["k_cache"], st["v_cache"], st["mask"]
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)

    def one(step, units=None):
        nonlocal ws
        inp = step_inputs(wl, step)
        res = oracle.decode_step(inp["q"], k, v, mask, inp["new_k"], inp["new_v"], ws, wl.W,
                                 wl.scale, units=units)
        nxt = res["next_slot"].copy()
        nxt[nxt < -1] = -1  # units outside a sample: no write at the next step
        ws = nxt

    warm = []
    for s in range(max(1, args.warmup)):
        t0 = time.perf_counter()
        one(s)
        warm.append(time.perf_counter() - t0)
    full_s = statistics.median(warm)
    units = None
    if args.steps * full_s > args.reference_seconds:
        n = max(1, int(wl.units * args.reference_seconds / (args.steps * full_s)))
        rng = np.random.default_rng(0)
        units = np.sort(rng.choice(wl.units, size=min(n, wl.units), replace=False)).astype(np.int32)
    t0 = time.perf_counter()
    for s in range(args.steps):
        one(max(1, args.warmup) + s, units)
    dt = time.perf_counter() - t0
    if units is None:
        sec_per_step = dt / args.steps
        sample = (f"{args.steps} whole decode steps (all {wl.units} (b,kvh) units each), "
                  f"after {max(1, args.warmup)} whole warm-up steps")
    else:
        sec_per_step = dt / args.steps * wl.units / units.size
        sample = (f"{units.size} of {wl.units} (b,kvh) units per step (the whole steps would "
                  f"not fit in {args.reference_seconds:.0f} s), time scaled by "
                  f"{wl.units / units.size:.1f} to a full step")
    value = 1.0 / sec_per_step
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, world),
        "timed_region_s": dt,
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129 * 2**20


def l2_note(wl, layers=1) -> str:
    """How the timed steps relate to L2 (no flush between steps in any case)."""
    kv = wl.B * wl.Hkv * wl.S * wl.d * 2 * 2
    if kv > L2_BYTES:
        return f"inputs larger than L2 (K/V caches {kv / 2**20:.0f} MiB > 129 MiB); no flush between steps"
    if kv * layers > L2_BYTES:
        return (f"{layers} caches of {kv / 2**20:.1f} MiB stepped in turn "
                f"({kv * layers / 2**20:.0f} MiB > 129 MiB L2); no flush between steps")
    need = L2_BYTES // kv + 1
    return (f"inputs fit in L2 (K/V caches {kv / 2**20:.2f} MiB) and stay resident between "
            f"steps (no flush); --layers {need} or more steps that many caches in turn so that "
            "each step reads DRAM")


def workload_config(wl, world, layers=1, plan=None):
    cfg = {"workload": wl.name, "layers": layers, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
           "S": wl.S, "W": wl.W, "live": list(wl.live) if isinstance(wl.live, tuple) else wl.live,
           "description": wl.description,
           "l2": l2_note(wl, layers),
           "parallelism": f"replicas x{world} (disjoint sequences, no collective)"}
    if plan is not None:
        cfg["launch_plan"] = plan
    return cfg


def bench_lf(args, wl):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import decode_kv_cache_step_gb300 as lf
    from decode_kv_cache_step_gb300 import build as lfbuild
    if not lfbuild.up_to_date() and rank == 0:
        lfbuild.build()
    if world > 1:
        torch.distributed.barrier()
    lf.load_library()

    # Each rank runs its own B sequences of the recipe (weak scaling).
    from decode_kv_cache_step_gb300.sharding import max_over_ranks, weak_shard
    shard = weak_shard(wl, rank, world)
    host = initial_state(wl, batch_offset=shard.batch_offset)
    lengths = host["lengths"]
    k = bf16_dev(host["k_cache"], device)
    v = bf16_dev(host["v_cache"], device)
    mask = torch.from_numpy(host["mask"]).to(device)
    pool = []
    for s in range(8):
        inp = step_inputs(wl, s, batch_offset=shard.batch_offset, full_batch=shard.full_batch)
        pool.append({kk: bf16_dev(vv, device) for kk, vv in inp.items()})
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device=device)
    # Layer 0 holds the generated caches; further layers (--layers) are copies,
    # each with its own mask and write/next slot pair.
    L = args.layers
    layers = [(k, v, mask)] + [(k.clone(), v.clone(), mask.clone()) for _ in range(L - 1)]
    slots = [[torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32, device=device),
              torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device=device)] for _ in range(L)]
    # The timed steps replay CUDA graphs: one token through all L layers per
    # replay, or at one layer a run of n_graph consecutive steps (the largest
    # divisor of K up to 32), so that the host's launch rate does not set
    # the step rate of the small workloads (--eager: one Python call per step).
    use_graph = not args.eager
    n_graph = 1
    if use_graph and L == 1:
        n_graph = max(n for n in range(1, 33) if args.steps % n == 0)
    stream = torch.cuda.Stream(device) if use_graph else torch.cuda.current_stream(device)

    def step_eager(i, layer_ids=None):
        p = pool[i % len(pool)]
        for li in (range(L) if layer_ids is None else layer_ids):
            kk, vv, mm = layers[li]
            lf.decode_step(p["q"], kk, vv, mm, p["new_k"], p["new_v"], slots[li][i % 2], out,
                           slots[li][(i + 1) % 2], wl.W, wl.scale, stream=stream)

    lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)
    lf.profile_collect(lf.LF_KERNEL_SCORE)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            if i == args.warmup - 1:
                lf.profile_enable(True)   # count the kernels of one step
            step_eager(i)
    torch.cuda.synchronize()
    lf.profile_enable(False)
    n_step = lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)[1]
    n_score = lf.profile_collect(lf.LF_KERNEL_SCORE)[1]
    # Kernel launches per layer step: the decode-step kernel, plus the
    # scoring kernel when the step takes the split finish (long units).
    launches_per_layer = 1 + (n_score // max(n_step, 1))
    if lf.device_errors(stream) != 0:
        raise RuntimeError("device error word set during warm-up")

    graphs = []
    if use_graph:
        # Graph `parity` holds the n_graph steps that start at a step of that
        # parity (step j uses write/next slot buffers j % 2 and (j + 1) % 2 of
        # every layer), so that replays continue the token sequence.
        for parity in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(n_graph):
                    step_eager(args.warmup + parity + j)
            graphs.append(g)
        torch.cuda.synchronize()

    def replay_from(i0, n):
        # n steps from step i0 (n a multiple of n_graph)
        for b in range(n // n_graph):
            graphs[(i0 + b * n_graph) % 2].replay()

    if use_graph:
        # First replays (graph upload) outside the timed region; an even
        # number of steps keeps the slot parity of the token sequence.
        with torch.cuda.stream(stream):
            replay_from(0, 2 * n_graph)
        torch.cuda.synchronize()

    # ---------------------------------------------------------- device-timed
    clocks = ClockSampler(local)
    time.sleep(0.3)
    lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)
    lf.profile_collect(lf.LF_KERNEL_SCORE)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Pass 1 (value): K steps back to back, events around the whole loop only,
    # so consecutive launches overlap through programmatic dependent launch.
    t_wall0 = clocks.mark()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        if use_graph:
            replay_from(0, args.steps)
        else:
            for i in range(args.steps):
                step_eager(args.warmup + i)
        ev1.record(stream)
    torch.cuda.synchronize()
    ms_total = ev0.elapsed_time(ev1)
    # Pass 2 (roofline): K more steps, one call each, with the library's CUDA
    # events around every launch, on the launching stream, for the kernel's
    # own duration (layers > 1: graph replay time / launches).
    score_ms = 0.0
    if use_graph and L > 1:
        kern_ms, kern_n = ms_total, args.steps * L   # graph replays: launches back to back
    else:
        lf.profile_enable(True)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step_eager(args.warmup + args.steps + i)
        torch.cuda.synchronize()
        lf.profile_enable(False)
        kern_ms, kern_n = lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)
        score_ms = lf.profile_collect(lf.LF_KERNEL_SCORE)[0]
    t_wall1 = clocks.mark()
    ms_total = max_over_ranks(ms_total, device)
    if lf.device_errors(stream) != 0:
        raise RuntimeError("device error word set during the timed steps")

    # ------------------------------------- score + eviction over attention
    overhead = None
    if not args.no_overhead:
        n_o = max(20, min(args.steps, 200))
        att_ws = slots[0][0].clone()
        lf.profile_collect(lf.LF_KERNEL_ATTENTION)
        lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)
        lf.profile_collect(lf.LF_KERNEL_SCORE)
        torch.cuda.synchronize()
        lf.profile_enable(True)
        with torch.cuda.stream(stream):
            for i in range(n_o):
                step_eager(i, layer_ids=[0])
            for i in range(n_o):
                p = pool[i % len(pool)]
                lf.decode_attention(p["q"], k, v, mask, p["new_k"], p["new_v"], att_ws, out,
                                    wl.scale, stream=stream)
        torch.cuda.synchronize()
        lf.profile_enable(False)
        f_ms, f_n = lf.profile_collect(lf.LF_KERNEL_DECODE_STEP)
        fs_ms = lf.profile_collect(lf.LF_KERNEL_SCORE)[0]
        a_ms, a_n = lf.profile_collect(lf.LF_KERNEL_ATTENTION)
        f_avg, a_avg = (f_ms + fs_ms) / max(f_n, 1), a_ms / max(a_n, 1)
        overhead = {"fused_kernel_ms": f_avg, "attention_only_kernel_ms": a_avg,
                    "frac": (f_avg - a_avg) / a_avg if a_avg > 0 else None, "launches": n_o,
                    "score_kernel_ms": fs_ms / max(f_n, 1),
                    "how": "same resident caches; lf_decode_step (its kernels, the scoring "
                           "kernel included when the step splits its finish) vs "
                           "lf_decode_attention (same pipeline without row norms, score terms, "
                           "ageing, selection)"}

        # Per-token cost of two eviction policies on the same caches, back to
        # back steps (events around each loop only): LongFlow's eviction at
        # every step against compressing every K = 128 steps (K - 1 steps of
        # attention alone, then one step returning and masking K slots).
        K = 128
        n_p = 2 * K
        topk_out = torch.empty((wl.B, wl.Hkv, K), dtype=torch.int32, device=device)
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        with torch.cuda.stream(stream):
            pe[0].record(stream)
            for i in range(n_p):
                step_eager(i, layer_ids=[0])
            pe[1].record(stream)
            for i in range(n_p):
                p = pool[i % len(pool)]
                if i % K == K - 1:
                    lf.decode_step_ex(p["q"], k, v, mask, p["new_k"], p["new_v"], att_ws, out,
                                      topk_out, wl.W, wl.scale, k=K,
                                      flags=lf.LF_STEP_MASK_EVICTED, stream=stream)
                else:
                    lf.decode_attention(p["q"], k, v, mask, p["new_k"], p["new_v"], att_ws, out,
                                        wl.scale, stream=stream)
            pe[2].record(stream)
        torch.cuda.synchronize()
        every = pe[0].elapsed_time(pe[1]) / n_p
        periodic = pe[1].elapsed_time(pe[2]) / n_p
        overhead["policy_ms_per_step"] = {
            "every_step_argmin": every, f"every_{K}_steps_top{K}": periodic,
            "frac": (every - periodic) / periodic if periodic > 0 else None}

    # ------------------------------------------------------ end to end (host)
    pin = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
    hpool = []
    for s in range(8):
        inp = step_inputs(wl, s, batch_offset=shard.batch_offset, full_batch=shard.full_batch)
        hpool.append({kk: pin(vv).view(torch.bfloat16) for kk, vv in inp.items()})
    h_out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16).pin_memory()
    # Per layer two pinned slot buffers take turns: step i writes into slot
    # buffer i % 2 and returns the next slot in the other one.
    h_slots = [[torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32).pin_memory(),
                torch.empty((wl.B, wl.Hkv), dtype=torch.int32).pin_memory()] for _ in range(L)]

    # The serving loop's call: one prepared step per layer, input set and
    # slot parity (lf_step_prepare once; each step is one lf_step_run).
    handles = [[lf.PreparedStep(hpool[j]["q"], kk, vv, mm, hpool[j]["new_k"], hpool[j]["new_v"],
                                h_slots[li][j % 2], h_out, h_slots[li][(j + 1) % 2], wl.W,
                                wl.scale, stream=stream)
                for j in range(len(hpool))] for li, (kk, vv, mm) in enumerate(layers)]

    def e2e_step(i):
        for hl in handles:
            hl[i % len(hpool)].run()
        stream.synchronize()

    # The per-call entry point (argument checks, plan and pointer queries
    # every call), for comparison.
    def e2e_step_unprepared(i):
        p = hpool[i % len(hpool)]
        for li, (kk, vv, mm) in enumerate(layers):
            lf.decode_step_host(p["q"], kk, vv, mm, p["new_k"], p["new_v"], h_slots[li][i % 2],
                                h_out, h_slots[li][(i + 1) % 2], wl.W, wl.scale, stream=stream)
        stream.synchronize()

    def timed(fn, i0):
        n_warm = min(args.warmup, 6)
        for i in range(i0, i0 + n_warm):
            fn(i)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for i in range(i0 + n_warm, i0 + n_warm + args.steps):
            fn(i)
        return max_over_ranks(time.perf_counter() - t0, device), i0 + n_warm + args.steps

    # Both loops continue the same token sequence (even step counts keep the
    # slot parity of each loop's first step).
    e2e_s, i_next = timed(e2e_step, 0)
    e2e_plain_s, _ = timed(e2e_step_unprepared, i_next + (i_next % 2))
    if lf.device_errors(stream) != 0 or any(h.errors() for hl in handles for h in hl):
        raise RuntimeError("device error word set during the end-to-end steps")
    for hl in handles:
        for h in hl:
            h.close()
    clocks.stop()
    h2d = L * ((wl.B * wl.Hq * wl.d * 2) + 2 * (wl.B * wl.Hkv * wl.d * 2) + wl.B * wl.Hkv * 4)
    d2h = L * (wl.B * wl.Hq * wl.d * 2 + wl.B * wl.Hkv * 4)

    # ------------------------------------------------------------ CPU oracle
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        n, secs, threads, times = run_oracle_steps(wl, host, max_seconds=args.cpu_seconds,
                                                   max_steps=50, nthreads=args.cpu_threads)
        cpu = {"value": n / secs / L, "unit": "steps/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} full decode step(s) of one layer of the same workload, fp64, "
                         f"{threads} OpenMP threads" + (f", divided by {L} layers" if L > 1 else ""),
               "median_step_s": float(np.median(times)), "cpu_model": cpu_model()}

    if rank != 0:
        return 0

    ms_per_step = ms_total / args.steps
    value = world * args.steps / (ms_total / 1e3)
    alg_launch = algorithmic_bytes(wl, lengths)
    alg = alg_launch * L
    # A split finish adds the scoring kernel to every step: the roofline then
    # covers both kernels of the step (one event pair around the two, which
    # overlap; the scoring kernel has no time of its own).
    split = launches_per_layer > 1
    kern_avg_ms = (kern_ms + score_ms) / max(kern_n, 1)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = alg_launch / (kern_avg_ms / 1e3) / 1e9
    step_gbs = alg / (ms_per_step / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "value_timing": (f"CUDA events around K steps replayed as CUDA graphs of {n_graph} "
                         f"step(s) x {L} layer(s); consecutive launches overlap through "
                         f"programmatic dependent launch") if use_graph else
                        "CUDA events around K steps, one Python call per step",
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(wl, world, L,
                                  plan=lf.step_plan(wl.B, wl.Hq, wl.Hkv, wl.d, wl.S)),
        "hbm": {"algorithmic_bytes_per_step": alg, "achieved_gbs": step_gbs,
                "frac_of_measured_peak": step_gbs / peak, "frac_of_8000_gbs": step_gbs / 8000.0,
                "peak_kind": peak_kind},
        "roofline": {"kernel": "lf_decode_step_kernel" + (" + lf_score_kernel" if split else ""),
                     "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     # the committed counters cover one full-batch launch of one workload
                     "traffic": (committed_traffic() if L == 1 and not split and world == 1
                                 and wl.name == PROFILE_WORKLOAD and args.batch is None
                                 else None),
                     "algorithmic_bytes_per_launch": alg_launch,
                     "avg_launch_ms": kern_avg_ms, "launches": kern_n,
                     "score_kernel_avg_ms": score_ms / max(kern_n, 1) if split else None,
                     "timing": ("library CUDA events around each launch, second timed pass "
                                "of K steps, one call each") if L == 1 else
                               "CUDA-graph replay time / launches",
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "overhead_vs_attention_only": overhead,
        "cpu_baseline": cpu,
        "e2e": {"value": world * args.steps / e2e_s, "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "PreparedStep.run (lf_step_run) per layer on pinned host buffers: the "
                       "kernel reads the step's inputs and writes its results in host memory "
                       "in place over the host link (LF_HOST_ZEROCOPY=0 stages them with "
                       "copies); stream sync every step, the next slot read back from host "
                       "memory as the next step's write slot",
                "per_call_entry_value": world * args.steps / e2e_plain_s,
                "per_call_entry": "lf_decode_step_host per layer (checks, plan and pointer "
                                  "queries every call), same buffers"},
        "gpu_launches": args.steps * L * launches_per_layer,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="run the first BATCH sequences of the workload (small profiling cases)")
    ap.add_argument("--impl", default="lf", choices=["lf", "reference"])
    ap.add_argument("--reference-seconds", type=float, default=150.0,
                    help="--impl reference: time budget of the K timed oracle steps; whole "
                         "steps when they fit, else a sample of units per step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="OpenMP threads of the CPU baseline (0: all)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overhead", action="store_true",
                    help="skip the attention-only comparison")
    ap.add_argument("--layers", type=int, default=1,
                    help="decode through L layers' caches per step (one CUDA graph per "
                         "token when L > 1); Qwen3-8B has 36")
    ap.add_argument("--eager", action="store_true",
                    help="time one Python call per step (per layer) instead of replaying "
                         "CUDA graphs of the steps")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps, always
    wl = WORKLOADS[args.workload]
    if args.batch is not None:
        wl = wl.with_batch(args.batch)
    if args.impl == "reference":
        return bench_reference(args, wl)
    return bench_lf(args, wl)


if __name__ == "__main__":
    sys.exit(main())
