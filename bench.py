#!/usr/bin/env python3
"""Benchmark: one forward of chunk-wise paged self-attention per step.

A step is the whole hot path for one forward of the long-window workload:
for each of the 40 layers, the slot-mapping KV write of the current chunk
into that layer's pools, then paged attention of the chunk's queries over the
visible window (1 sink frame + 16 recent frames, 26520 keys) for both CFG
branches.  The per-forward host metadata is built once (as the pages build it
once per forward for all layers) and is not part of the device timing; the
``e2e`` figure re-uploads it every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line (rank 0).  Timing: CUDA events on the launching stream,
barrier + synchronize on both sides, max over ranks.  Inputs are larger than
L2 (every layer has its own 1.1 GB of pools, so each layer's keys are cold).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# Host<->device copies overlap kernels only when their stream and the compute stream use different hardware
# work queues.  With the default 8 queues the end-to-end step was seen to run its uploads after the compute
# (the step time was exactly the sum of the two) in some processes and not in others; asking for the
# maximum makes a shared queue unlikely.  Set before CUDA starts; it configures this process's context only.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")


METRIC = "paged attention TFLOP/s (% bf16 peak); KV-write GB/s (% HBM peak)"
DEFAULT_WORKLOAD = "long-window-40L-bf16"


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def visible_pairs(meta) -> int:
    """Visible (query, key) pairs summed over rows, from the library's host metadata."""
    return pairs_from_segments(meta.query_start_loc, meta.seq_lens, meta.segments)


def pairs_from_segments(query_start_loc, seq_lens, segments) -> int:
    """Visible (query, key) pairs of rows given their (q_start, q_end, kv_end, mode) segments
    (mode 1 = full); a row without segments sees all of its keys."""
    pairs = 0
    for b in range(len(seq_lens)):
        sq = int(query_start_loc[b + 1] - query_start_loc[b])
        L = int(seq_lens[b])
        off = L - sq
        segs = segments[b] if segments is not None and segments[b] else [(off, L, L, 1)]
        for (s, e, kv_end, mode) in segs:
            n = e - s
            kv_end = min(kv_end, L)
            if mode == 1:
                pairs += n * kv_end
            else:
                shift = kv_end - n
                # rows r = 0..n-1 see min(kv_end, r + shift + 1) keys (clamped at 0)
                for r in range(n):
                    pairs += max(0, min(kv_end, r + shift + 1))
    return pairs


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle leg


_ORACLE_CASES: dict = {}


def _oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        info = threadpool_info()
        return max(int(i.get("num_threads", 1)) for i in info) if info else (os.cpu_count() or 1)
    except Exception:
        return os.cpu_count() or 1


def cpu_oracle_sample(w, budget_s: float = 12.0, max_heads: int | None = None, rows: int = 1) -> dict:
    """Time the float32 oracle on the workload's layer 0: the first ``rows`` rows (CFG branches), whole
    (row, head) pairs in order until ``budget_s`` of CPU time has passed (all of them when it is None)."""
    import dataclasses

    import numpy as np

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import pagedattn as pa
    from paged_kv_cache_181_gb300 import synth
    from tests import cases

    w1 = dataclasses.replace(w, batch=rows, layers=1)
    oc = _ORACLE_CASES.get(w1.name, {}).get(rows)
    if oc is None:  # inputs and pools are built once, outside the timed region
        d = synth.draw(w1, 0, "cpu")
        oc = cases.oracle_metadata(w1)
        cases.oracle_pools(w1, d, oc)
        _ORACLE_CASES.setdefault(w1.name, {})[rows] = oc
    n_heads = w1.num_heads if max_heads is None else min(max_heads, w1.num_heads)
    units = [(b, h) for b in range(rows) for h in range(n_heads)]
    flops_per_unit = [pa.attention_flops(oc.qsl[b:b + 2] - oc.qsl[b], oc.seq_lens[b:b + 1],
                                         None if oc.segments is None else oc.segments[b:b + 1], 1, w1.head_dim)
                      for b in range(rows)]
    flops = 0
    done = 0
    t0 = time.perf_counter()
    for b, h in units:
        sample = {(b, h): np.arange(w1.q_len)}
        pa.paged_attention(oc.q, oc.k_pool, oc.v_pool, oc.table, oc.qsl, oc.seq_lens, w1.head_dim ** -0.5,
                           w1.block_size, oc.segments, dtype=np.float32, sample=sample)
        flops += flops_per_unit[b]
        done += 1
        if budget_s is not None and time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    row_txt = "row 0" if rows == 1 else f"rows 0-{rows - 1}"
    what = (f"{row_txt}, all {w1.num_heads} heads" if done == len(units) and n_heads == w1.num_heads
            else f"{row_txt}, {done} of {rows * w1.num_heads} (row, head) pairs")
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": f"{w.name}: layer 0, {what}, {w1.q_len} queries x {int(oc.seq_lens[0])} keys each, "
                      f"float32 NumPy oracle ({dt:.1f} s)", "seconds": dt}


def cpu_write_sample(w) -> dict:
    """Time the oracle's KV write (oracle.pagedattn.kv_write, a row-by-row copy) of one layer's current chunk,
    K and V, on the workload's own bytes: 16-bit values are handled as uint16 bit patterns, so the bytes
    moved are those of the GPU write.  The pools are touched once before the timed write."""
    import numpy as np
    import torch

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import pagedattn as pa
    from paged_kv_cache_181_gb300 import synth
    from tests import cases

    oc = cases.oracle_metadata(w)
    d = synth.draw(w, 0, "cpu")
    def host_bits(t):
        t = t.contiguous()
        return t.numpy() if w.dtype == "f32" else t.view(torch.int16).numpy().view(np.uint16)

    k, v = host_bits(d.k_cur), host_bits(d.v_cur)
    bits = k.dtype
    n_slots = w.pool_blocks * w.block_size
    kp = np.zeros((n_slots, w.num_kv_heads, w.head_dim), dtype=bits)
    vp = np.zeros_like(kp)
    pa.kv_write(kp, oc.slots, k)
    pa.kv_write(vp, oc.slots, v)
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        pa.kv_write(kp, oc.slots, k)
        pa.kv_write(vp, oc.slots, v)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    tq = len(oc.slots)
    nbytes = tq * 2 * (2 * k[0].nbytes) + tq * 8
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{w.name}: one layer's write, {tq} tokens x K and V rows of {k[0].nbytes} B into "
                      f"{n_slots}-slot pools, oracle kv_write (one Python-level row copy per row, one thread; "
                      f"median of 3: {dt * 1e3:.1f} ms)", "seconds": dt}


def workload_config(w, world: int) -> dict:
    row_bytes = w.num_kv_heads * w.head_dim * (2 if w.dtype != "f32" else 4)
    return {"workload": w.name, "layers": w.layers, "batch": w.batch, "heads": w.num_heads,
            "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "q_len": w.q_len, "block_size": w.block_size,
            "history_tokens": w.history_tokens, "window_chunks": w.window_chunks, "sink_chunks": w.sink_chunks,
            "chunk_tokens": w.chunk_tokens, "pool_blocks_per_layer": w.pool_blocks,
            "l2": "inputs larger than L2: each layer reads its own %.2f GB of pools" %
                  (2 * w.pool_blocks * 16 * row_bytes / 1e9),
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    from paged_kv_cache_181_gb300 import configs

    w = configs.ALL[args.workload]
    budget = max(1.0, min(8.0, 120.0 / max(1, args.steps)))  # the whole run stays within a few minutes
    for _ in range(args.warmup):
        cpu_oracle_sample(w, budget_s=0.5, max_heads=1)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_oracle_sample(w, budget_s=budget))
    elapsed = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, world) | {"sample": vals[0]["sample"]},
        "cpu_baseline": {k: vals[0][k] for k in ("unit", "cores", "kind", "sample")} | {"value": v},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU leg


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    from paged_kv_cache_181_gb300 import _lib, configs, workload

    w = configs.ALL[args.workload]
    peaks = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workload.build_case(w, device=dev, poison=False)
    meta = case.meta
    layers = case.layers
    pairs = visible_pairs(meta)
    flops_per_layer = 4 * w.head_dim * w.num_heads * pairs
    tq = int(meta.query_start_loc[-1])
    row_bytes = w.num_kv_heads * w.head_dim * (2 if w.dtype != "f32" else 4)
    write_bytes_per_layer = tq * 2 * (2 * row_bytes) + tq * 8  # read + write of K and V rows, plus the slot ids
    stream = torch.cuda.current_stream()

    fused = not args.two_call

    def step():
        case.step(stream=stream, fused=fused)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # Per-launch durations over separate instrumented steps (events between launches).
    ev_w = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]
    ev_a = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]
    write_ms, attn_ms, launch_log = [], [], []
    # KV write: a burst of one write per layer (a single ~20 us launch is too short to time alone), each
    # write into its own cold layer pool, replayed from a CUDA graph.
    write_avg = graph_burst_ms([lambda l=l: case.write(l) for l in range(layers)], stream)
    # The launches of one step as it runs them: the fused write + attention, or (two-call form) the
    # attention call after its layer's write.
    for _ in range(1):
        for l in range(layers):
            if not fused:
                ev_w[l][0].record(stream)
                case.write(l, stream=stream)
                ev_w[l][1].record(stream)
            ev_a[l][0].record(stream)
            if fused:
                case.write_attend(l, stream=stream)
            else:
                case.attend(l, stream=stream)
            attn_launches_l = _lib.last_launches()
            ev_a[l][1].record(stream)
            launch_log.append(attn_launches_l)
        torch.cuda.synchronize()
        if not fused:
            write_ms += [ev_w[l][0].elapsed_time(ev_w[l][1]) for l in range(layers)]
        attn_launches = launch_log[-layers:]
        attn_ms += [ev_a[l][0].elapsed_time(ev_a[l][1]) for l in range(layers)]

    # Timed region: K whole steps.  Each layer's attention call is bracketed by events inside the timed
    # steps themselves, so the per-call duration behind the roofline is taken at the clock the step runs at
    # (steps started from idle run faster until the power cap settles).
    ev_t = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(layers)]
            for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        start.record(stream)
        for k in range(args.steps):
            for l in range(layers):
                if not fused:
                    case.write(l, stream=stream)
                ev_t[k][l][0].record(stream)
                if fused:
                    case.write_attend(l, stream=stream)
                else:
                    case.attend(l, stream=stream)
                ev_t[k][l][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    attn_ms = [e0.elapsed_time(e1) for row in ev_t for e0, e1 in row]
    ms = max_over_ranks(start.elapsed_time(end), world)
    ms_step = ms / args.steps
    total_flops = flops_per_layer * layers * world
    value = total_flops / (ms_step * 1e-3) / 1e12

    split_plan = dict(zip(("splits", "whole_items"), _lib.last_split_plan()))
    attn_avg = statistics.mean(attn_ms)
    attn_tflops = flops_per_layer / (attn_avg * 1e-3) / 1e12
    write_gbs = write_bytes_per_layer / (write_avg * 1e-3) / 1e9
    # Per layer: the attention launch (+ combine when split), plus the write launch in the two-call form.
    launches_per_step = sum((0 if fused else 1) + attn_launches[l] for l in range(layers))

    traffic = read_traffic(w.name)

    # The same step captured once in a CUDA graph and replayed.
    graph = measure_graph(case, args.steps, fused, ms_step) if not args.no_graph else None

    # The other way to run the same forward (two calls per layer, or the fused call).
    alt = measure_alt_step(case, stream, args.steps, ms_step, not fused) if not args.no_alt else None

    # Paged vs contiguous K/V on the same data (the pages' gather-then-attend path).
    kv_layout = measure_kv_layout(case, stream, attn_avg, row_bytes) if not args.no_kv_layout else None

    # Packed heterogeneous rows: one call over rows of different shapes and query offsets.
    packed_rows = measure_packed(stream, peaks) if not args.no_packed else None
    split_kv = measure_split_kv(stream, peaks) if not args.no_packed else None

    # e2e: inputs from pinned host memory every step, outputs back to the host.
    e2e = run_e2e(case, args, world, stream, fused, local) if not args.no_e2e else None

    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1), shapes of 832x480 frames)",
        "config": workload_config(w, world),
        # The attention calls are timed inside the 40-layer step (about 53 ms of back-to-back launches at the
        # power cap), so the denominator is the sustained dense bf16 figure; the burst fraction is given beside it.
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_tflops_sustained"], "traffic": traffic,
                     "peak_source": f"{peaks['source']} bf16 dense, sustained (the kernel is timed inside the step)",
                     "frac_of_burst": attn_tflops / peaks["bf16_tflops"], "burst_peak": peaks["bf16_tflops"],
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                     "kernel": "paged attention (fused with the layer's KV write)" if fused else "paged attention",
                     "ms_per_launch": attn_avg,
                     "algorithmic_flops_per_launch": flops_per_layer},
        "kv_write": {"bound": "hbm", "achieved": write_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": write_gbs / peaks["hbm_gbs"], "ms_per_launch": write_avg,
                     "algorithmic_bytes_per_launch": write_bytes_per_layer,
                     "traffic": read_traffic(w.name, "kv_write_long_window.md", WRITE_KERNEL_REV),
                     "traffic_note": "DRAM read + write during one launch (ncu); the rest of the pool rows is "
                                     "written back from L2 after it",
                     "kernel": "paged_kv_write (standalone launch; inside the fused call it overlaps the attention)"},
        "gpu_launches": args.steps * launches_per_step,
        "step_api": "paged_kv_write_attn per layer (write fused into the attention launch)" if fused
                    else "paged_kv_write + paged_attn_varlen per layer",
        "clocks": clocks.summary(),
    }
    if e2e is not None:
        result["e2e"] = e2e
    if kv_layout is not None:
        result["kv_layout"] = kv_layout
    if graph is not None:
        result["graph"] = graph
    if alt is not None:
        result["fused" if not fused else "two_call"] = alt
    if packed_rows is not None:
        result["packed_rows"] = packed_rows
    if split_kv is not None:
        result["split_kv"] = split_kv
    # Every workload at full size, one layer each (the long-window entry is this step's own figures).
    if not args.no_workloads:
        wl = {w.name: {
            "attention": {"api": result["step_api"], "ms_per_call": attn_avg,
                          "algorithmic_flops_per_call": flops_per_layer, "tflops": attn_tflops,
                          "frac_of_burst": attn_tflops / peaks["bf16_tflops"],
                          "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                          "launches_per_call": attn_launches[0], "split_plan": split_plan,
                          "l2": "each layer reads its own pools (cold)", "dtype": w.dtype},
            "kv_write": {"us_per_launch": write_avg * 1e3, "algorithmic_bytes_per_launch": write_bytes_per_layer,
                         "gbs": write_gbs, "frac_of_hbm": write_gbs / peaks["hbm_gbs"],
                         "burst_launches": layers, "timing": "burst replayed from one CUDA graph",
                         "row_bytes": row_bytes, "rows": 2 * tq},
            "clocks": result["clocks"]}}
        for name in OTHER_WORKLOADS:
            if name != w.name:
                wl[name] = measure_workload(name, stream, peaks)
        result["workloads"] = wl
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from paged_kv_cache_181_gb300 import configs as _cfg

        main_cpu = cpu_oracle_sample(w)
        extra = [cpu_oracle_sample(_cfg.ONE_FRAME, budget_s=None, rows=2),
                 cpu_oracle_sample(_cfg.MIXED_MASK, budget_s=None, rows=2),
                 cpu_write_sample(_cfg.LONG_WINDOW), cpu_write_sample(_cfg.MIXED_MASK)]
        result["cpu_baseline"] = {k: v for k, v in main_cpu.items() if k != "seconds"} | {
            "cases": [{k: v for k, v in c.items() if k != "seconds"} for c in extra]}
    if rank == 0:
        print(json.dumps(result), flush=True)


KERNEL_REV = "tc-v16"


def measure_graph(case, steps: int, fused: bool, main_ms_step: float) -> dict:
    """The forward step captured in a CUDA graph (every layer's launches) and replayed ``steps`` times."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        case.step(fused=fused)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        case.step(fused=fused)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = 4 * case.w.head_dim * case.w.num_heads * visible_pairs(case.meta) * case.layers
    del g
    return {"ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "main_step_ms": main_ms_step, "note": "same step, all launches replayed from one CUDA graph"}


def measure_alt_step(case, stream, steps: int, main_ms_step: float, fused: bool) -> dict:
    """Forward steps through the other API: paged_kv_write_attn (one launch per layer) or two calls."""
    import torch

    for _ in range(3):
        case.step(stream=stream, fused=fused)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        case.step(stream=stream, fused=fused)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = 4 * case.w.head_dim * case.w.num_heads * visible_pairs(case.meta) * case.layers
    return {"api": "paged_kv_write_attn per layer" if fused else "paged_kv_write + paged_attn_varlen per layer",
            "ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "main_step_ms": main_ms_step, "main_over_this": main_ms_step / ms}


def _time_packed(pc, stream, flags: int, reps: int) -> float:
    import torch

    for _ in range(3):
        pc.attend(flags=flags, stream=stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    for e0, e1 in ev:
        e0.record(stream)
        pc.attend(flags=flags, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)


def measure_split_kv(stream, peaks: dict, reps: int = 20) -> dict:
    """Split-KV + combine where it matters: few (row, head) units over a long window."""
    import torch

    from paged_kv_cache_181_gb300 import _lib, configs, packed

    pb = configs.PACKED_FEW_HEADS
    pc = packed.build_packed(pb, poison=False)
    flops = 4 * pb.head_dim * pb.num_heads * pairs_from_segments(pc.qsl_host, pc.seq_lens_host, pc.segments)
    ms_auto = _time_packed(pc, stream, 0, reps)
    launches = _lib.last_launches()
    ms_one = _time_packed(pc, stream, _lib.PKV_NO_SPLIT, reps)
    res = {"workload": pb.name, "ms_split": ms_auto, "ms_no_split": ms_one, "speedup": ms_one / ms_auto,
           "launches_split": launches, "tflops_split": flops / (ms_auto * 1e-3) / 1e12,
           "tflops_no_split": flops / (ms_one * 1e-3) / 1e12}
    del pc
    torch.cuda.empty_cache()
    return res


def measure_packed(stream, peaks: dict, reps: int = 10) -> dict:
    """TFLOP/s of one attention call over the packed heterogeneous rows (6 rows of the 832x480 model)."""
    import torch

    from paged_kv_cache_181_gb300 import configs, packed

    pb = configs.PACKED_MIXED
    pc = packed.build_packed(pb, poison=False)
    flops = 4 * pb.head_dim * pb.num_heads * pairs_from_segments(pc.qsl_host, pc.seq_lens_host, pc.segments)
    ms = _time_packed(pc, stream, 0, reps)
    tflops = flops / (ms * 1e-3) / 1e12
    res = {"workload": pb.name, "rows": len(pb.rows), "ms_per_launch": ms, "algorithmic_flops_per_launch": flops,
           "achieved": tflops, "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
           "rows_desc": [[r.query_len, r.seq_len, r.kv_start_pos, len(r.spans)] for r in pb.rows]}
    del pc
    torch.cuda.empty_cache()
    return res


def measure_kv_layout(case, stream, step_call_ms: float, row_bytes: int) -> dict:
    """Per layer: the block gather of the visible window into staging buffers, the same attention on the
    staged (contiguous) K/V, and the re-gather of the current chunk's blocks only (history kept staged)."""
    import torch

    layers = case.layers
    st = case.make_staging()
    for l in range(min(3, layers)):
        case.stage(l, st, stream=stream)
        case.attend_contiguous(l, st, stream=stream)
    torch.cuda.synchronize()

    def burst(fn, reps=3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        out = []
        for _ in range(reps):
            e0.record(stream)
            for l in range(layers):
                fn(l)
            e1.record(stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) / layers)
        return statistics.median(out)

    gather_ms = burst(lambda l: case.stage(l, st, stream=stream))
    regather_ms = burst(lambda l: case.stage(l, st, reuse_history=True, stream=stream))
    # The same attention call (paged_attn_varlen) on the pools and on staged K/V, alternating layer by layer so
    # both run at the same clock: events around each launch, every layer staged just before.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(layers)]
    contig_ms, paged_only_ms = [], []
    for _ in range(2):
        for l in range(layers):
            case.stage(l, st, stream=stream)
            ev[l][0].record(stream)
            case.attend(l, stream=stream)
            ev[l][1].record(stream)
            ev[l][2].record(stream)
            case.attend_contiguous(l, st, stream=stream)
            ev[l][3].record(stream)
        torch.cuda.synchronize()
        paged_only_ms += [ev[l][0].elapsed_time(ev[l][1]) for l in range(layers)]
        contig_ms += [ev[l][2].elapsed_time(ev[l][3]) for l in range(layers)]
    contig = statistics.mean(contig_ms)
    paged_ms = statistics.mean(paged_only_ms)
    staged_rows = case.w.batch * st.used_blocks * case.w.block_size
    chunk_rows = case.w.batch * (st.used_blocks - st.first_block) * case.w.block_size
    res = {
        "paged_attn_ms": paged_ms, "contiguous_attn_ms": contig, "paged_over_contiguous": paged_ms / contig,
        "api": "paged_attn_varlen on the pools and on the staged window, alternating per layer",
        "fused_step_call_ms": step_call_ms,
        "gather_ms": gather_ms, "gather_gbs": staged_rows * row_bytes * 4 / (gather_ms * 1e-3) / 1e9,
        "regather_chunk_ms": regather_ms, "regather_blocks_per_row": st.used_blocks - st.first_block,
        "gather_then_attend_ms": gather_ms + contig, "regather_then_attend_ms": regather_ms + contig,
        "chunk_rows": chunk_rows,
    }
    del st
    torch.cuda.empty_cache()
    return res


OTHER_WORKLOADS = ("tiny-f32", "one-frame-bf16", "one-frame-partial-bf16", "gqa-action-bf16", "mixed-mask-bf16",
                   "long-window-f32-1L")


def fp32_fma_peak_tflops() -> float:
    """CUDA-core fp32 rate: SMs x 128 FMA lanes x 2 FLOP x the maximum SM clock (nominal, not measured)."""
    import torch

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    return props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12


def _l2_bytes() -> int:
    import torch

    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 2**20


def graph_burst_ms(calls, stream, reps: int = 3) -> float:
    """Per-call device time of a burst of short launches: the calls are captured once in a CUDA graph and the
    graph is replayed between two events, so the host's per-call submission cost (the Python binding takes
    longer to submit a launch than a 20-40 us write takes to run) does not leave the GPU idle between them."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for c in calls:
            c()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / len(calls))
    del g
    return statistics.median(per)


def measure_write_burst(w, case, stream, reps: int = 3) -> dict:
    """Standalone KV write of one workload: a burst of R launches, each from its own source tensors into its
    own pool pair, so that no launch finds its bytes in L2 (R x bytes >= 4 x L2); per launch = burst / R,
    replayed from a CUDA graph (graph_burst_ms)."""
    import torch

    row_bytes = w.num_kv_heads * w.head_dim * (2 if w.dtype != "f32" else 4)
    tq = int(case.meta.query_start_loc[-1])
    nbytes = tq * 2 * (2 * row_bytes) + tq * 8
    n_sets = max(4, min(64, -(-4 * _l2_bytes() // nbytes)))
    sets = [(case.k_new[0], case.v_new[0], case.k_pools[0], case.v_pools[0])]
    for _ in range(n_sets - 1):
        sets.append((case.k_new[0].clone(), case.v_new[0].clone(), torch.empty_like(case.k_pools[0]),
                     torch.empty_like(case.v_pools[0])))
    from paged_kv_cache_181_gb300 import _lib

    calls = [lambda k=k, v=v, kp=kp, vp=vp: _lib.paged_kv_write(k, v, case.slots, kp, vp) for k, v, kp, vp in sets]
    ms = graph_burst_ms(calls, stream, reps)
    del sets, calls
    torch.cuda.empty_cache()
    return {"us_per_launch": ms * 1e3, "algorithmic_bytes_per_launch": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "burst_launches": n_sets, "timing": "burst replayed from one CUDA graph", "row_bytes": row_bytes,
            "rows": 2 * tq}


def measure_workload(name: str, stream, peaks: dict, reps: int = 20) -> dict:
    """One workload at full size, one layer: the fused write + attention call timed per launch (an L2 flush
    before each, events around it), its split plan, and the standalone write (measure_write_burst)."""
    import torch

    from paged_kv_cache_181_gb300 import _lib, configs, workload

    w = (configs.ALL | configs.VARIANTS)[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    case = workload.build_case(w, device=dev, layers=1, data_device=dev)
    flops = 4 * w.head_dim * w.num_heads * visible_pairs(case.meta)
    flush = torch.empty(4 * _l2_bytes(), dtype=torch.uint8, device=dev)
    for _ in range(3):
        case.write_attend(0, stream=stream)
    torch.cuda.synchronize()
    plan = _lib.last_split_plan()
    launches = _lib.last_launches()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        # The same work for about 0.6 s first, so that the 200 ms clock samples land while it runs.
        t_end = time.perf_counter() + 0.6
        while time.perf_counter() < t_end:
            flush.zero_()
            case.write_attend(0, stream=stream)
            torch.cuda.synchronize()
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            case.write_attend(0, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        wr = measure_write_burst(w, case, stream)
    del flush
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    tflops = flops / (ms * 1e-3) / 1e12
    att_peak = {"frac_of_burst": tflops / peaks["bf16_tflops"],
                "frac_of_sustained": tflops / peaks["bf16_tflops_sustained"]} if w.dtype != "f32" else {
        "frac_of_fp32_fma": tflops / fp32_fma_peak_tflops(),
        "peak_note": "fp32 runs on the CUDA cores: the denominator is the nominal fp32 FMA rate"}
    res = {
        "attention": {"api": "paged_kv_write_attn (fused write + attention), one layer", "ms_per_call": ms,
                      "algorithmic_flops_per_call": flops, "tflops": tflops} | att_peak | {
                      "launches_per_call": launches, "split_plan": {"splits": plan[0], "whole_items": plan[1]},
                      "l2": "flushed before each timed call", "dtype": w.dtype},
        "kv_write": wr | {"frac_of_hbm": wr["gbs"] / peaks["hbm_gbs"]},
        "clocks": clk.summary(),
    }
    del case
    torch.cuda.empty_cache()
    return res


WRITE_KERNEL_REV = "w-v2"


def read_traffic(workload_name: str, summary: str = "attn_tc_long_window.md", rev: str | None = None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken of this kernel revision."""
    import re

    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    m = re.search(r"traffic: workload=(\S+) rev=(\S+) bytes_per_launch=(\d+)", open(path).read())
    if not m or m.group(1) != workload_name or m.group(2) != (KERNEL_REV if rev is None else rev):
        return None
    return int(m.group(3))


def run_e2e(case, args, world, stream, fused: bool, gpu_index: int = 0):
    """The same forward through the public API with every input coming from pinned host memory.

    Per step: the per-forward metadata and every layer's Q, new K and new V are copied host -> device on a
    copy stream, each layer's write + attention runs on the compute stream as soon as its inputs have
    landed, and each layer's output is copied device -> host on a third stream as soon as it is ready.
    Alternate steps use two device copies of the inputs and outputs, so that a step's uploads never wait
    for the previous step's compute of the same layer (uploads run slower while the attention runs on
    some machines; with one copy that coupled the two streams layer by layer), and a step's last read-backs
    overlap the next step's first layers.  Every copy of every timed step is inside the timed region.
    """
    import torch

    layers = case.layers
    host_q = [t.cpu().pin_memory() for t in case.q]
    host_k = [t.cpu().pin_memory() for t in case.k_new]
    host_v = [t.cpu().pin_memory() for t in case.v_new]
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in case.out]
    meta_host = [t.cpu().pin_memory() for t in (case.slots, case.block_table, case.query_start_loc, case.seq_lens)]
    meta_dev = [case.slots, case.block_table, case.query_start_loc, case.seq_lens]
    if case.segs is not None:
        meta_host += [case.segs.cpu().pin_memory(), case.seg_start.cpu().pin_memory()]
        meta_dev += [case.segs, case.seg_start]
    h2d = sum(t.numel() * t.element_size() for t in host_q + host_k + host_v + meta_host)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    up = torch.cuda.Stream()
    # K and V of a layer upload on streams of their own beside Q's, so that copies can use more than one copy
    # engine at a time.
    up_k, up_v = torch.cuda.Stream(), torch.cuda.Stream()
    down = torch.cuda.Stream()
    # Two device sets of the per-layer inputs and outputs, used by alternate steps.
    io_sets = [(case.q, case.k_new, case.v_new, case.out),
               ([t.clone() for t in case.q], [t.clone() for t in case.k_new], [t.clone() for t in case.v_new],
                [torch.empty_like(t) for t in case.out])]
    landed = [[torch.cuda.Event() for _ in range(layers)] for _ in range(2)]
    computed = [[torch.cuda.Event() for _ in range(layers)] for _ in range(2)]
    fetched = [[torch.cuda.Event() for _ in range(layers)] for _ in range(2)]
    # Two device copies of the per-forward metadata, used by alternate steps, so that a step's metadata
    # upload does not wait for the previous step's last layer.
    meta_sets = [meta_dev, [t.clone() for t in meta_dev]]
    meta_landed = [torch.cuda.Event(), torch.cuda.Event()]
    meta_free = [torch.cuda.Event(), torch.cuda.Event()]
    names = ["slots", "block_table", "query_start_loc", "seq_lens", "segs", "seg_start"]
    step_no = [0]

    # Each layer's uploads timed between events on the copy stream (after its wait): their sum in a step
    # against upload_ms_alone says whether the uploads slow down while the attention runs.
    up_t = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]
    # Each layer's compute timed the same way (after its waits): their sum against the step says whether the
    # compute itself slowed down or waited for its inputs.
    cp_t = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]

    def e2e_step(last: bool = True):
        k = step_no[0] % 2
        step_no[0] += 1
        q_d, k_d, v_d, o_d = io_sets[k]
        with torch.cuda.stream(up):
            up.wait_event(meta_free[k])
            for hd, dd in zip(meta_host, meta_sets[k]):
                dd.copy_(hd, non_blocking=True)
            meta_landed[k].record(up)
            for l in range(layers):
                up.wait_event(computed[k][l])  # the step before last no longer reads this set's inputs
                up_t[l][0].record(up)
                up_k.wait_stream(up)
                up_v.wait_stream(up)
                q_d[l].copy_(host_q[l], non_blocking=True)
                with torch.cuda.stream(up_k):
                    k_d[l].copy_(host_k[l], non_blocking=True)
                with torch.cuda.stream(up_v):
                    v_d[l].copy_(host_v[l], non_blocking=True)
                up.wait_stream(up_k)
                up.wait_stream(up_v)
                landed[k][l].record(up)
                up_t[l][1].record(up)
        for name, t in zip(names, meta_sets[k]):
            setattr(case, name, t)
        case.q, case.k_new, case.v_new, case.out = q_d, k_d, v_d, o_d
        stream.wait_event(meta_landed[k])
        for l in range(layers):
            stream.wait_event(landed[k][l])
            stream.wait_event(fetched[k][l])  # this set's output of the step before last has been read back
            cp_t[l][0].record(stream)
            if fused:
                case.write_attend(l, stream=stream)
            else:
                case.write(l, stream=stream)
                case.attend(l, stream=stream)
            computed[k][l].record(stream)
            cp_t[l][1].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[k][l])
                host_out[l].copy_(o_d[l], non_blocking=True)
                fetched[k][l].record(down)
        meta_free[k].record(stream)
        if last:  # the timed region ends with every output on the host
            stream.wait_stream(down)

    for ev in fetched[0] + fetched[1] + computed[0] + computed[1] + meta_free:
        ev.record(stream)
    e2e_step()
    e2e_step()
    torch.cuda.synchronize()
    # One step's uploads alone, without compute: the host->device bandwidth this machine gives, so that an
    # upload-bound step shows as such beside the overlapped one.  Taken right before and right after the
    # timed steps: the link's speed was seen to change over time with no GPU work of this process running.
    def uploads_alone_ms() -> float:
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(up):
            u0.record(up)
            for hd, dd in zip(meta_host, meta_sets[0]):
                dd.copy_(hd, non_blocking=True)
            for l in range(layers):
                io_sets[0][0][l].copy_(host_q[l], non_blocking=True)
                io_sets[0][1][l].copy_(host_k[l], non_blocking=True)
                io_sets[0][2][l].copy_(host_v[l], non_blocking=True)
            u1.record(up)
        torch.cuda.synchronize()
        return u0.elapsed_time(u1)

    upload_ms = uploads_alone_ms()
    steps = max(1, min(args.steps, 5))
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:  # clocks while copies and compute overlap (power draw differs)
        start.record(stream)
        up.wait_event(start)  # no upload of the timed steps starts before the clock does
        # Steps are pipelined: a step's last read-backs overlap the next step's first layers (its output
        # buffers are the other set's); the last step ends with every read-back done.
        marks = [start]
        for i in range(steps):
            e2e_step(last=i == steps - 1)
            marks.append(torch.cuda.Event(enable_timing=True))
            marks[-1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    upload_ms_after = uploads_alone_ms()
    # The case's tensors again those it started with (the second set and its events go with this function).
    case.q, case.k_new, case.v_new, case.out = io_sets[0]
    for name, t in zip(names, meta_sets[0]):
        setattr(case, name, t)
    ms = max_over_ranks(start.elapsed_time(end), world) / steps
    flops = 4 * case.w.head_dim * case.w.num_heads * visible_pairs(case.meta) * layers * world
    api = "paged_kv_write_attn" if fused else "paged_kv_write + paged_attn_varlen"
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "api": f"{api} per layer, inputs from pinned host memory",
            "upload_ms_alone": upload_ms, "h2d_gbs_alone": h2d / (upload_ms * 1e-3) / 1e9,
            "h2d_gbs_alone_after": h2d / (upload_ms_after * 1e-3) / 1e9,
            "step_ms": [round(marks[i].elapsed_time(marks[i + 1]), 3) for i in range(steps)],
            "upload_ms_in_last_step": sum(up_t[l][0].elapsed_time(up_t[l][1]) for l in range(layers)),
            "compute_ms_in_last_step": sum(cp_t[l][0].elapsed_time(cp_t[l][1]) for l in range(layers)),
            "cuda_device_max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS"),
            "clocks": clk.summary()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kv-layout", action="store_true", help="skip the paged vs contiguous K/V comparison")
    ap.add_argument("--no-packed", action="store_true", help="skip the packed heterogeneous rows measurement")
    ap.add_argument("--two-call", action="store_true",
                    help="time the forward as paged_kv_write + paged_attn_varlen per layer (default: the fused call)")
    ap.add_argument("--no-alt", action="store_true", help="skip timing the other API for comparison")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay measurement")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' per-call figures")
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
