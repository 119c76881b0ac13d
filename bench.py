#!/usr/bin/env python3
"""Benchmark of paged MLA decode (libmla) on one GB300, or N replicas.

A step is one mla_decode call over one batch of synthetic input: the main
attention kernel and the LSE-combine kernel, launched through the C ABI.  The
split-KV plan is computed once per decode step and shared by every layer, so
it is timed apart (its own pass of K planner calls) and reported beside the
value, as is a plan + decode pass.  The default workload is the large-batch
128-head decode (batch 16, s_q 1, h_q 128, 4096 cached tokens per sequence,
576/512 latent dims, 64-token pages, random page order).

Timing: W untimed warm-up steps, then exactly K steps between CUDA events on
the launching stream, with a device synchronise (and, for N > 1, a barrier)
on both sides; rank 0 prints one JSON line.  L2 is defeated by rotating
input sets whose total size is well above the L2 capacity, so every step
reads its cache pages from HBM.  Per-kernel durations come from events
recorded between the launches of a second pass.

--impl reference times the fp64 CPU oracle on the host cores instead (the
only other arm there is: the pages ship no implementation).

--workload sparse_b64_h128_l131072_k2048 measures sparse decode instead
(mla_decode_sparse with 2048 listed positions per entry of a 128K-token
context; plans over the counts made beforehand), with rotating query/position
sets.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_decode_attention_07_gb300 import workloads as W  # noqa: E402

METRIC = "MLA decode TFLOP/s, KV GB/s and % of GB300 roofline per call (1 GPU)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = "b16_h128_l4096"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attend_traffic.json")
SPARSE_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "sparse_traffic.json")
DECODE_SRC = os.path.join(ROOT, "mla_decode_attention_07_gb300", "csrc", "mla_decode_sm103.cu")
NARROW_SRC = os.path.join(ROOT, "mla_decode_attention_07_gb300", "csrc", "mla_decode_narrow_sm103.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(W.WORKLOADS) + sorted(W.SPARSE_WORKLOADS) +
                    sorted(W.GEMM_WORKLOADS) + sorted(W.PROLOGUE_WORKLOADS) +
                    sorted(W.ATTENTION_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline leg")
    return ap.parse_args(argv)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_max(value: float, world: int) -> float:
    """Max over ranks of a per-rank float (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def roofline_times(w: W.Workload, peaks):
    t_mem = w.bytes() / (peaks["hbm_gbs"] * 1e9)
    t_flop = w.flops() / (peaks["bf16_tflops"] * 1e12)
    return t_mem, t_flop


def kernel_code_sha(path: str) -> str:
    """sha256 of a CUDA source with its // comments and blank lines removed:
    the code the counters were taken on, independent of comment edits."""
    lines = []
    for line in open(path, encoding="utf-8").read().splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code.strip():
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def traffic_per_launch(workload: str, path: str = TRAFFIC_FILE, src: str = DECODE_SRC):
    """DRAM bytes per launch from the committed ncu summary: the record taken
    on this workload, if the source of the kernel that ran is unchanged since
    (a file holds one record, or a list under "records")."""
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            data = json.load(f)
        recs = data.get("records", [data])
        sha = kernel_code_sha(src)
        for rec in recs:
            if rec.get("workload") == workload and rec.get("code_sha256") == sha:
                return float(rec["dram_bytes_per_launch_full_workload"])
        return None
    except Exception:
        return None


def physical_gpu_index(logical: int) -> int:
    """nvidia-smi numbers GPUs physically; map through CUDA_VISIBLE_DEVICES."""
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if logical < len(vis) and vis[logical].isdigit():
        return int(vis[logical])
    return logical


class ClockSampler:
    """nvidia-smi sampling (every 200 ms) while the GPU is under load."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(w: W.Workload, inp, budget_s: float):
    """The oracle as it stands, on this host's cores, over whole passes of the
    workload (or a row sample when one pass would exceed the budget)."""
    import oracle
    threads = oracle.default_threads()
    rows_all = np.array([(b, i, h) for b in range(w.batch) for i in range(w.s_q)
                         for h in range(w.h_q)], dtype=np.int32)
    keys = inp.cache_seqlens.astype(np.int64)
    flops_row = {}
    # one small calibration call, then size the sample to the budget
    t0 = time.perf_counter()
    cal = rows_all[: max(1, min(len(rows_all), 8))]
    oracle.mla_decode_rows(inp, cal, nthreads=threads)
    dt = max(1e-6, time.perf_counter() - t0)

    def fl(rows):
        tot = 0.0
        for b, i, h in rows:
            n = max(0, int(keys[b]) - w.s_q + 1 + int(i))
            tot += 2.0 * (W.D_QK + W.D_V) * n
        return tot
    rate = fl(cal) / dt
    total_fl = w.flops()
    if total_fl / rate <= budget_s:
        sample, desc = rows_all, "full workload"
    else:
        n = max(1, int(len(rows_all) * budget_s * rate / total_fl / 1.2))
        rng = np.random.default_rng(0)
        sample = rows_all[np.sort(rng.choice(len(rows_all), size=n, replace=False))]
        desc = f"{n} of {len(rows_all)} query rows, seeded random"
    sfl = fl(sample)
    passes, spent = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.mla_decode_rows(inp, sample, nthreads=threads)
        spent += time.perf_counter() - t0
        passes += 1
        if spent >= 0.5 * budget_s or passes >= 50:
            break
    value = sfl * passes / spent / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{desc}, {passes} pass(es), {spent:.1f} s, fp64 C oracle"}


def make_sets(torch, w: W.Workload, dev, l2_bytes: int):
    """Input sets rotated between steps; total bytes > 2.5 x L2."""
    per_set = w.bytes()
    n = max(2, math.ceil(2.5 * l2_bytes / per_set))
    seqlens = w.seqlens()
    sets = []
    host0 = None
    for k in range(n):
        inp = w.make() if k == 0 else W.make_inputs(w.seed + 7919 * k, w.batch, w.s_q, w.h_q,
                                                    seqlens)
        if k == 0:
            host0 = inp
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        sets.append(dict(q=t(inp.q.view(np.int16)).view(torch.bfloat16),
                         kv=t(inp.kv_cache.view(np.int16)).view(torch.bfloat16),
                         bt=t(inp.block_table), sl=t(inp.cache_seqlens)))
    return sets, host0


def run_ours(args):
    import torch
    from mla_decode_attention_07_gb300 import libmla

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    libmla.load()
    w = W.WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    sets, host0 = make_sets(torch, w, dev, l2)
    B, s_q, h_q = w.batch, w.s_q, w.h_q
    out = torch.empty((B, s_q, h_q, W.D_V), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, h_q, s_q), dtype=torch.float32, device=dev)
    meta, ws = libmla.alloc_plan_and_workspace(B, s_q, h_q, dev.index)
    stream = torch.cuda.current_stream(dev)
    scale = W.SOFTMAX_SCALE

    # every input set has the same sequence lengths, so one plan serves them
    # all, as one plan serves every layer of a decode step
    libmla.mla_decode_plan(sets[0]["sl"], s_q, h_q, meta, stream)

    def step(k):
        s = sets[k % len(sets)]
        libmla.mla_decode(s["q"], s["kv"], s["bt"], s["sl"], meta, out, lse, scale, ws, stream)

    def step_with_plan(k):
        s = sets[k % len(sets)]
        libmla.mla_decode_plan(s["sl"], s_q, h_q, meta, stream)
        libmla.mla_decode(s["q"], s["kv"], s["bt"], s["sl"], meta, out, lse, scale, ws, stream)

    def step_split(k, evs):
        # the same launches with an event between each pair (this breaks the
        # programmatic overlap of consecutive launches, so it is only used for
        # the per-kernel durations)
        s = sets[k % len(sets)]
        evs[0].record(stream)
        libmla.mla_decode_plan(s["sl"], s_q, h_q, meta, stream)
        evs[1].record(stream)
        libmla.mla_decode_attend(s["q"], s["kv"], s["bt"], s["sl"], meta, out, lse, scale, ws,
                                 stream)
        evs[2].record(stream)
        libmla.mla_decode_combine(B, s_q, h_q, meta, out, lse, ws, stream)
        evs[3].record(stream)

    def timed(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    for k in range(max(3, args.warmup)):
        step_with_plan(k)
        step(k)
    torch.cuda.synchronize()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error during warm-up: {libmla.mla_strerror(rc)}")

    # Keep the GPU busy ~1.5 s under the clock sampler, then the timed region.
    sampler = ClockSampler(physical_gpu_index(dev.index))
    sampler.start()
    t_end = time.perf_counter() + 1.5
    k = 0
    while time.perf_counter() < t_end:
        for _ in range(50):
            step(k)
            k += 1
        torch.cuda.synchronize()

    K = args.steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    start.record(stream)
    for i in range(K):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_total = start.elapsed_time(end)
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: {libmla.mla_strerror(rc)}")
    # the planner alone and plan + decode, each over its own pass of K calls
    plan_alone_ms = timed(lambda i: libmla.mla_decode_plan(sets[i % len(sets)]["sl"], s_q, h_q,
                                                           meta, stream), K)
    with_plan_ms = aggregate_max(timed(step_with_plan, K), world)
    # the same mla_decode calls replayed from a CUDA graph: the host's per-call
    # issue cost (Python, argument checks, tensor maps) is then out of the
    # timed region, as in a decode step captured whole
    gwin = len(sets) * max(1, math.ceil(20 / len(sets)))

    def step_on(k, st):
        s = sets[k % len(sets)]
        libmla.mla_decode(s["q"], s["kv"], s["bt"], s["sl"], meta, out, lse, scale, ws, st)

    graph_ms = aggregate_max(_timed_graph(torch, stream, step_on, K, gwin), world)
    # per-kernel durations over a further pass of K steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        step_split(i, evs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    plan_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
    attend_us = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) * 1e3
    combine_us = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) * 1e3
    ms_total = aggregate_max(ms_total, world)
    ms_step = ms_total / K

    # End to end through the public API from pinned host buffers: every step
    # copies q, block table and sequence lengths in, runs mla_decode_plan +
    # mla_decode, and copies out and lse back.  The cache pages stay resident
    # on the device (they are the model's state, not a per-step input); sets
    # still rotate for L2.  Steps are pipelined the way a serving loop would
    # run them: the inputs of the next step and the results of the previous
    # one move on two copy streams while a step computes (each input set has
    # its own out/lse and tile metadata, and a set is refilled only after its
    # last step's results are copied out), and a window of steps is captured
    # once as a CUDA graph so that the host issues one launch per window.  A
    # step's plan needs only its sequence lengths, so it runs on the input
    # stream right after they land, while the previous step decodes.  A
    # step's inputs sit in one pinned buffer and its out + lse in one device
    # buffer, so each direction is a single copy.
    def packed(parts, device=None, pin=False):
        """One byte buffer holding several tensors (16-byte aligned views), so
        that a step's inputs, or its outputs, move in a single copy."""
        offs, off = [], 0
        for shape, dt in parts:
            off = (off + 15) // 16 * 16
            offs.append(off)
            off += int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = []
        for (shape, dt), o in zip(parts, offs):
            n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
            views.append(buf[o:o + n].view(dt).view(shape))
        return buf, views

    in_parts = [(tuple(sets[0]["q"].shape), torch.bfloat16), (tuple(sets[0]["bt"].shape), torch.int32),
                (tuple(sets[0]["sl"].shape), torch.int32)]
    out_parts = [(tuple(out.shape), torch.bfloat16), (tuple(lse.shape), torch.float32)]
    h_in, (hq, hbt, hsl) = packed(in_parts, pin=True)
    hq.copy_(torch.from_numpy(np.ascontiguousarray(host0.q.view(np.int16))).view(torch.bfloat16))
    hbt.copy_(torch.from_numpy(host0.block_table))
    hsl.copy_(torch.from_numpy(host0.cache_seqlens))
    win = min(4 * len(sets), 32)     # steps per captured window
    ns = min(len(sets), win)         # input sets the window rotates through
    d_in = [packed(in_parts, device=dev) for _ in range(ns)]
    d_res = [packed(out_parts, device=dev) for _ in range(ns)]
    d_meta = [torch.empty_like(meta) for _ in range(ns)]   # one plan buffer per input set
    h_res = [packed(out_parts, pin=True)[0] for _ in range(ns)]
    h2d = hq.numel() * 2 + hbt.numel() * 4 + hsl.numel() * 4
    d2h = out.numel() * 2 + lse.numel() * 4

    def e2e_window(cap):
        """Enqueue `win` pipelined steps on `cap` (and two copy streams that
        fork from and join back into it).  Per step: one host-to-device copy
        of the packed inputs and the plan (input stream), the decode (`cap`),
        one device-to-host copy of the packed out + lse (output stream)."""
        hs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        hs.wait_stream(cap)
        ds.wait_stream(cap)
        ready = [torch.cuda.Event() for _ in range(win)]
        done = [torch.cuda.Event() for _ in range(win)]
        back = [torch.cuda.Event() for _ in range(win)]
        for j in range(win):
            i = j % ns
            kv = sets[i]["kv"]
            ibuf, (q_i, bt_i, sl_i) = d_in[i]
            rbuf, (out_i, lse_i) = d_res[i]
            with torch.cuda.stream(hs):
                if j >= ns:
                    hs.wait_event(done[j - ns])
                ibuf.copy_(h_in, non_blocking=True)
                libmla.mla_decode_plan(sl_i, s_q, h_q, d_meta[i], hs)
                ready[j].record(hs)
            cap.wait_event(ready[j])
            if j >= ns:
                cap.wait_event(back[j - ns])
            libmla.mla_decode(q_i, kv, bt_i, sl_i, d_meta[i], out_i, lse_i, scale, ws, cap)
            done[j].record(cap)
            with torch.cuda.stream(ds):
                ds.wait_event(done[j])
                h_res[i].copy_(rbuf, non_blocking=True)
                back[j].record(ds)
        cap.wait_stream(hs)
        cap.wait_stream(ds)

    e2e_mode = f"pipelined, {win}-step CUDA graph"
    graph = None
    try:
        cap = torch.cuda.Stream(dev)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            e2e_window(cap)
    except Exception as ex:   # capture unavailable: the same window issued directly
        graph = None
        e2e_mode = f"pipelined, {win} steps issued directly (graph capture failed: {type(ex).__name__})"
    torch.cuda.synchronize()

    def run_window():
        if graph is not None:
            graph.replay()
        else:
            e2e_window(stream)

    for _ in range(2):
        run_window()
    torch.cuda.synchronize()
    reps = max(1, K // win)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e_start.record(stream)
    for _ in range(reps):
        run_window()
    e_end.record(stream)
    torch.cuda.synchronize()
    e2e_ms = aggregate_max(e_start.elapsed_time(e_end), world) / (reps * win)
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in e2e region: {libmla.mla_strerror(rc)}")

    flops = w.flops() * world
    tflops = flops / (ms_step * 1e-3) / 1e12
    kv_bytes = float(w.seqlens().astype(np.int64).sum()) * W.D_QK * 2
    t_mem, t_flop = roofline_times(w, peaks)
    roof_s = max(t_mem, t_flop)
    bound = "hbm" if t_mem >= t_flop else "tensor"
    attend_s = attend_us * 1e-6
    if bound == "hbm":
        achieved = w.bytes() / attend_s / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = w.flops() / attend_s / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    # which decode kernel this shape runs (the narrow one: <= 32 query rows)
    narrow = libmla.mla_decode_kernel_kind(B, s_q, h_q, int(sets[0]["bt"].shape[1]), dev.index) == 1
    kernel_name = "mla_decode_narrow_kernel (attend)" if narrow else "mla_decode_kernel (attend)"
    traffic = traffic_per_launch(w.name, TRAFFIC_FILE, NARROW_SRC if narrow else DECODE_SRC)

    result = {
        "metric": METRIC,
        "value": round(tflops, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 normals rounded to bf16; random page order)",
        "config": {"workload": w.name, "batch": B, "s_q": s_q, "h_q": h_q,
                   "seqlen": int(w.seqlen) if w.seqlen else "ragged", "d_qk": W.D_QK,
                   "d_v": W.D_V, "page": W.PAGE, "softmax_scale": scale,
                   "l2": f"rotating {len(sets)} input sets of {w.bytes() / 1e6:.1f} MB "
                         f"(> 2.5 x L2 {l2 / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_call": round(ms_step * 1e3, 3),
        "graph_us_per_call": round(graph_ms * 1e3, 3),
        "graph_note": f"the same calls replayed from a {gwin}-call CUDA graph (host issue cost "
                      "out of the timed region); value is the calls issued one by one",
        "kv_gbs": round(kv_bytes * world / (ms_step * 1e-3) / 1e9, 1),
        "roofline_pct": round(100.0 * roof_s / (ms_step * 1e-3), 2),
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_name,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured"
                     else "fallback"},
        "kernels_us": {"plan": round(plan_us, 3), "attend": round(attend_us, 3),
                       "combine": round(combine_us, 3)},
        "gpu_launches": 2 * K,
        "kernels_note": "per-kernel durations from a further pass of K steps with events "
                        "between launches; value is the pass without them (mla_decode: "
                        "attend + combine per step, the plan computed once beforehand)",
        "plan": {"us_per_call": round(plan_alone_ms * 1e3, 3),
                 "note": "mla_decode_plan alone, K calls back to back; one plan serves every "
                         "layer of a decode step"},
        "plan_and_decode": {"us_per_step": round(with_plan_ms * 1e3, 3),
                            "value": round(w.flops() * world / (with_plan_ms * 1e-3) / 1e12, 3),
                            "unit": "TFLOP/s",
                            "roofline_pct": round(100.0 * roof_s / (with_plan_ms * 1e-3), 2)},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "steps": reps * win,
                "note": "every step: q/block_table/seqlens copied in from pinned host memory, "
                        "mla_decode_plan (on the input stream, overlapping the previous "
                        "step's decode) + mla_decode, out+lse copied back (one packed copy "
                        "each way); cache pages resident; " + e2e_mode},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, host0, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """fp64 CPU oracle timed as the comparison arm (rank 0 only)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = W.WORKLOADS[args.workload]
    inp = w.make()
    threads = oracle.default_threads()
    rows_all = np.array([(b, i, h) for b in range(w.batch) for i in range(w.s_q)
                         for h in range(w.h_q)], dtype=np.int32)
    keys = inp.cache_seqlens.astype(np.int64)

    def fl(rows):
        return sum(2.0 * (W.D_QK + W.D_V) * max(0, int(keys[b]) - w.s_q + 1 + int(i))
                   for b, i, _h in rows)
    cal = rows_all[:8]
    t0 = time.perf_counter()
    oracle.mla_decode_rows(inp, cal, nthreads=threads)
    rate = fl(cal) / max(1e-6, time.perf_counter() - t0)
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    n = int(min(len(rows_all), max(1, len(rows_all) * budget * rate / w.flops())))
    rng = np.random.default_rng(1)
    sample = rows_all if n >= len(rows_all) else \
        rows_all[np.sort(rng.choice(len(rows_all), size=n, replace=False))]
    sfl = fl(sample)
    for _ in range(args.warmup):
        oracle.mla_decode_rows(inp, sample, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mla_decode_rows(inp, sample, nthreads=threads)
    dt = time.perf_counter() - t0
    value = sfl * args.steps / dt / 1e12
    desc = "full workload" if n >= len(rows_all) else f"{n} of {len(rows_all)} query rows"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "s_q": w.s_q, "h_q": w.h_q,
                   "seqlen": int(w.seqlen) if w.seqlen else "ragged"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{desc} per step, fp64 C oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


SPARSE_METRIC = "MLA sparse decode TFLOP/s, gathered KV GB/s and % of GB300 roofline per call"


def sparse_sets(w, si, n):
    """Rotating (q, positions) sets over one cache pool: set 0 is the
    workload's own, the others redraw q and the positions."""
    seqlens = si.base.cache_seqlens
    out = [(si.base.q, si.indices, si.counts)]
    for k in range(1, n):
        sd = w.seed + 7919 * k
        q = W.normal_bf16(sd, W.TENSOR_Q, w.batch * w.h_q * W.D_QK).reshape(w.batch, 1, w.h_q,
                                                                           W.D_QK)
        idx, cnt = W.draw_indices(sd, seqlens, w.topk)
        out.append((q, idx, cnt))
    return out


def sparse_cpu_baseline(si, budget_s):
    """The oracle over a seeded row sample of the sparse workload."""
    import oracle
    threads = oracle.default_threads()
    B, h_q = si.base.batch, si.base.h_q
    rows_all = np.array([(b, h) for b in range(B) for h in range(h_q)], dtype=np.int32)
    per_row = 2.0 * (W.D_QK + W.D_V)
    fl = lambda rows: sum(per_row * int(si.counts[b]) for b, _h in rows)
    cal = rows_all[:16]
    t0 = time.perf_counter()
    oracle.mla_decode_sparse_rows(si, cal, nthreads=threads)
    rate = fl(cal) / max(1e-6, time.perf_counter() - t0)
    n = int(min(len(rows_all), max(16, budget_s * rate / per_row / max(1, si.topk) / 1.2)))
    rng = np.random.default_rng(0)
    sample = rows_all[np.sort(rng.choice(len(rows_all), size=n, replace=False))]
    passes, spent = 0, 0.0
    while spent < 0.5 * budget_s and passes < 50:
        t0 = time.perf_counter()
        oracle.mla_decode_sparse_rows(si, sample, nthreads=threads)
        spent += time.perf_counter() - t0
        passes += 1
    return {"value": fl(sample) * passes / spent / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{n} of {len(rows_all)} query rows, seeded random, {passes} pass(es), "
                      f"{spent:.1f} s, fp64 C oracle"}


def run_sparse(args):
    """Sparse decode on one GPU (or N replicas): one mla_decode_sparse call per
    step (its plan over the counts made beforehand), inputs resident, rotating
    position sets."""
    import torch
    from mla_decode_attention_07_gb300 import libmla

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    libmla.load()
    w = W.SPARSE_WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    si = w.make()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    kv = t(si.base.kv_cache.view(np.int16)).view(torch.bfloat16)
    bt, sl = t(si.base.block_table), t(si.base.cache_seqlens)
    sets = [dict(q=t(q.view(np.int16)).view(torch.bfloat16), idx=t(idx), cnt=t(cnt))
            for q, idx, cnt in sparse_sets(w, si, 4)]
    B, h_q = w.batch, w.h_q
    out = torch.empty((B, 1, h_q, W.D_V), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, h_q, 1), dtype=torch.float32, device=dev)
    meta, ws = libmla.alloc_plan_and_workspace(B, 1, h_q, dev.index)
    stream = torch.cuda.current_stream(dev)
    scale = W.SOFTMAX_SCALE
    # one plan per position set (over its counts), computed before the timed
    # region: a plan serves every layer of a decode step
    metas = []
    for st in sets:
        m, _ = libmla.alloc_plan_and_workspace(B, 1, h_q, dev.index)
        libmla.mla_decode_plan(st["cnt"], 1, h_q, m, stream)
        metas.append(m)

    def step(k, ev=None):
        st = sets[k % len(sets)]
        if ev:
            ev[0].record(stream)
            libmla.mla_decode_plan(st["cnt"], 1, h_q, meta, stream)
        if ev:
            ev[1].record(stream)
        libmla.mla_decode_sparse(st["q"], kv, bt, sl, st["idx"], st["cnt"],
                                 meta if ev else metas[k % len(sets)], out, lse, scale, ws,
                                 stream)
        if ev:
            ev[2].record(stream)

    for k in range(max(3, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error during warm-up: {libmla.mla_strerror(rc)}")
    sampler = ClockSampler(physical_gpu_index(dev.index))
    sampler.start()
    t_end = time.perf_counter() + 1.5
    k = 0
    while time.perf_counter() < t_end:
        for _ in range(20):
            step(k)
            k += 1
        torch.cuda.synchronize()
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for i in range(K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_step = aggregate_max(e0.elapsed_time(e1), world) / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        step(i, evs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: {libmla.mla_strerror(rc)}")
    plan_us = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
    call_us = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) * 1e3
    gbytes = w.bytes()
    achieved = gbytes / (call_us * 1e-6) / 1e9
    result = {
        "metric": SPARSE_METRIC,
        "value": round(w.flops() * world / (ms_step * 1e-3) / 1e12, 3),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 normals rounded to bf16; uniform random "
                "distinct positions; shared 8192-page pool)",
        "config": {"workload": w.name, "batch": B, "s_q": 1, "h_q": h_q, "seqlen": w.seqlen,
                   "topk": w.topk, "pool_pages": w.pool_pages,
                   "l2": "4 rotating query/position sets; each step gathers "
                         f"{w.keys() * W.D_QK * 2 / 1e6:.0f} MB of scattered rows from a "
                         f"{w.pool_pages * 64 * W.D_QK * 2 / 1e6:.0f} MB pool",
                   "parallelism": "single GPU" if world == 1 else f"{world} replicas"},
        "us_per_call": round(ms_step * 1e3, 3),
        "kv_gbs": round(w.keys() * W.D_QK * 2 / (ms_step * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic_per_launch(w.name, SPARSE_TRAFFIC_FILE),
                     "kernel": "mla_decode_sparse call (decode kernel + combine); traffic: "
                               "the decode kernel's DRAM bytes per launch",
                     "peak_source": peak_src},
        "kernels_us": {"plan": round(plan_us, 3), "decode_call": round(call_us, 3)},
        "gpu_launches": 2 * K,
        "kernels_note": "value: K mla_decode_sparse calls (decode kernel + combine) with "
                        "plans computed beforehand; plan and decode_call from a second pass "
                        "with events between launches",
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = sparse_cpu_baseline(si, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _timed_loop(torch, stream, fn, n):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(n):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _timed_graph(torch, stream, fn, n, window):
    """Average device time of one fn(i, stream) call: `window` calls are
    captured once as a CUDA graph and the graph is replayed between CUDA
    events, so the host's per-call issue cost (Python, argument checks,
    tensor-map encoding, the launch itself) is out of the timed region."""
    cap = torch.cuda.Stream(device=stream.device)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(window):
            fn(i, cap)
    stream.wait_stream(cap)
    reps = max(1, n // window)
    with torch.cuda.stream(stream):
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps * window)


def _single_gpu_setup():
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    return torch, world, rank, dev


GEMM_METRIC = "FP16 GEMM TFLOP/s and % of GB300 dense-bf16/fp16 tensor peak (1 GPU)"


def run_gemm(args):
    """C = A B (fp16 in, fp32 accumulate, fp16 out) through mla_gemm; cuBLAS
    (torch.matmul) timed on the same rotating input sets beside it."""
    torch, world, rank, dev = _single_gpu_setup()
    from mla_decode_attention_07_gb300 import libmla
    libmla.load()
    w = W.GEMM_WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    nsets = max(2, math.ceil(2.5 * l2 / w.bytes()))
    sets = []
    for k in range(nsets):
        if k == 0:
            a, b = w.make()
        else:
            a = W.normal_f16(w.seed + 7919 * k, W.TENSOR_GEMM_A, w.M * w.K).reshape(w.M, w.K)
            b = W.normal_f16(w.seed + 7919 * k, W.TENSOR_GEMM_B, w.K * w.N).reshape(w.K, w.N)
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x.view(np.int16))).to(dev).view(
            torch.float16)
        sets.append((t(a), t(b), torch.empty((w.M, w.N), dtype=torch.float16, device=dev)))
    stream = torch.cuda.current_stream(dev)

    def ours(i):
        a, b, c = sets[i % nsets]
        libmla.mla_gemm(a, b, c, stream)

    def cublas(i):
        a, b, c = sets[i % nsets]
        torch.matmul(a, b, out=c)

    for i in range(max(3, args.warmup)):
        ours(i)
        cublas(i)
    torch.cuda.synchronize()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error during warm-up: {libmla.mla_strerror(rc)}")
    sampler = ClockSampler(physical_gpu_index(dev.index))
    sampler.start()
    t_end = time.perf_counter() + 1.0
    i = 0
    while time.perf_counter() < t_end:
        for _ in range(20):
            ours(i)
            i += 1
        torch.cuda.synchronize()
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    ms = aggregate_max(_timed_loop(torch, stream, ours, K), world)
    ms_cublas = _timed_loop(torch, stream, cublas, K)
    clocks = sampler.stop()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: {libmla.mla_strerror(rc)}")
    tf = w.flops() / (ms * 1e-3) / 1e12
    tf_cublas = w.flops() / (ms_cublas * 1e-3) / 1e12
    # e2e: A and B copied in from pinned host memory, C copied back, per step
    ha = torch.from_numpy(np.ascontiguousarray(w.make()[0].view(np.int16))).pin_memory()
    hb = torch.from_numpy(np.ascontiguousarray(w.make()[1].view(np.int16))).pin_memory()
    hc = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
    da, db, dc = sets[0]

    def e2e(i):
        da.view(torch.int16).copy_(ha, non_blocking=True)
        db.view(torch.int16).copy_(hb, non_blocking=True)
        libmla.mla_gemm(da, db, dc, stream)
        hc.copy_(dc.view(torch.int16), non_blocking=True)

    for i in range(3):
        e2e(i)
    e2e_ms = aggregate_max(_timed_loop(torch, stream, e2e, max(5, K // 4)), world)
    result = {
        "metric": GEMM_METRIC, "value": round(tf * world, 3), "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) rounded to fp16)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "l2": f"rotating {nsets} input sets of {w.bytes() / 1e6:.1f} MB (> 2.5 x L2)",
                   "parallelism": "single GPU" if world == 1 else f"{world} replicas"},
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": None, "kernel": "mla_gemm_kernel",
                     "peak_source": f"{peak_src}: bf16 burst (fp16 has the same nominal rate)"},
        "cublas": {"value": round(tf_cublas, 3), "unit": "TFLOP/s",
                   "ms_per_step": round(ms_cublas, 5), "ratio": round(tf / tf_cublas, 4),
                   "how": "torch.matmul(out=) on the same rotating fp16 sets"},
        "gpu_launches": K,
        "e2e": {"value": round(w.flops() * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": 2 * 2 * w.M * w.K,
                "d2h_bytes_per_step": 2 * w.M * w.N},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        a0, b0 = w.make()
        rng = np.random.default_rng(0)
        n = 4096
        ent = np.stack([rng.integers(0, w.M, n), rng.integers(0, w.N, n)], 1).astype(np.int32)
        t0 = time.perf_counter()
        oracle.gemm_entries(a0, b0, 0, ent)
        dt = time.perf_counter() - t0
        result["cpu_baseline"] = {"value": 2.0 * w.K * n / dt / 1e12, "unit": "TFLOP/s",
                                  "cores": oracle.default_threads(), "kind": "oracle",
                                  "sample": f"{n} sampled entries of C, fp64 C oracle, "
                                            f"{dt:.2f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


PROLOGUE_METRIC = "MLA decode-step prologue (cache append + query absorption) GB/s and us per call"


def run_prologue(args):
    """mla_cache_append + mla_q_absorb per step at a decode workload's shape;
    input sets (W_UK of a layer each) rotate so that every step reads its
    weights from HBM, as successive layers do."""
    torch, world, rank, dev = _single_gpu_setup()
    from mla_decode_attention_07_gb300 import libmla
    libmla.load()
    w = W.PROLOGUE_WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20))
    p0 = w.make()
    bf = torch.bfloat16
    t = lambda x, dt=None: (torch.from_numpy(np.ascontiguousarray(x)).to(dev) if dt is None else
                            torch.from_numpy(np.ascontiguousarray(x.view(np.int16))).to(dev).view(dt))
    kv = t(p0.base.kv_cache, bf)
    bt, sl = t(p0.base.block_table), t(p0.base.cache_seqlens)
    nsets = max(2, math.ceil(2.5 * l2 / w.absorb_bytes()))
    sets = []
    for k in range(nsets):
        sd = w.seed + 7919 * k
        rows = w.batch * w.s_q
        sets.append(dict(
            new=t(W.normal_bf16(sd, W.TENSOR_KV_NEW, rows * W.D_QK).reshape(w.batch, w.s_q, W.D_QK), bf),
            qn=t(W.normal_bf16(sd, W.TENSOR_Q_NOPE, rows * w.h_q * W.D_NOPE).reshape(
                w.batch, w.s_q, w.h_q, W.D_NOPE), bf),
            qr=t(W.normal_bf16(sd, W.TENSOR_Q_ROPE, rows * w.h_q * W.D_ROPE).reshape(
                w.batch, w.s_q, w.h_q, W.D_ROPE), bf),
            wuk=t(W.scaled_normal_bf16(sd, W.TENSOR_W_UK, w.h_q * W.D_NOPE * W.D_C,
                                       W.D_NOPE ** -0.5).reshape(w.h_q, W.D_NOPE, W.D_C), bf),
            q=torch.empty((w.batch, w.s_q, w.h_q, W.D_QK), dtype=bf, device=dev)))
    stream = torch.cuda.current_stream(dev)

    def append(i, s=stream):
        st = sets[i % nsets]
        libmla.mla_cache_append(st["new"], kv, bt, sl, s)

    def absorb(i, s=stream):
        st = sets[i % nsets]
        libmla.mla_q_absorb(st["qn"], st["qr"], st["wuk"], st["q"], s)

    def step(i, s=stream):
        append(i, s)
        absorb(i, s)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error during warm-up: {libmla.mla_strerror(rc)}")
    sampler = ClockSampler(physical_gpu_index(dev.index))
    sampler.start()
    t_end = time.perf_counter() + 1.0     # load under the clock sampler
    i = 0
    while time.perf_counter() < t_end:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    # the calls replayed from CUDA graphs (device time); issued one by one
    # from Python beside it, where the host's issue cost can dominate
    window = nsets * max(1, math.ceil(20 / nsets))
    ms = aggregate_max(_timed_graph(torch, stream, step, K, window), world)
    ms_append = _timed_graph(torch, stream, append, K, window)
    ms_absorb = _timed_graph(torch, stream, absorb, K, window)
    host_ms = {"append": _timed_loop(torch, stream, append, K),
               "absorb": _timed_loop(torch, stream, absorb, K),
               "step": _timed_loop(torch, stream, step, K)}
    clocks = sampler.stop()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: {libmla.mla_strerror(rc)}")
    nbytes = w.absorb_bytes() + w.append_bytes()
    gbs = nbytes / (ms * 1e-3) / 1e9
    absorb_gbs = w.absorb_bytes() / (ms_absorb * 1e-3) / 1e9
    result = {
        "metric": PROLOGUE_METRIC, "value": round(gbs * world, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rows and queries, W_UK ~ N(0, 1/128), bf16)",
        "config": {"workload": w.name, "batch": w.batch, "s_q": w.s_q, "h_q": w.h_q,
                   "d_nope": W.D_NOPE, "d_c": W.D_C,
                   "l2": f"rotating {nsets} weight/query sets of {w.absorb_bytes() / 1e6:.1f} MB "
                         "(> 2.5 x L2)",
                   "parallelism": "single GPU" if world == 1 else f"{world} replicas"},
        "us_per_call": {"append": round(ms_append * 1e3, 3), "absorb": round(ms_absorb * 1e3, 3),
                        "step": round(ms * 1e3, 3)},
        "timing": f"CUDA events around replays of a {window}-call CUDA graph ({K} calls timed)",
        "host_issued_us_per_call": {k: round(v * 1e3, 3) for k, v in host_ms.items()},
        "roofline": {"bound": "hbm", "achieved": round(absorb_gbs, 2), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(absorb_gbs / peaks["hbm_gbs"], 4),
                     "traffic": None,
                     "kernel": "mla_absorb_kernel (with its rotary copy)",
                     "bytes_per_call": w.absorb_bytes(), "peak_source": peak_src},
        "absorb_tflops": round(w.absorb_flops() / (ms_absorb * 1e-3) / 1e12, 3),
        "gpu_launches": 2 * max(1, K // window) * window,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle's append + absorption over whole passes of the workload
        import oracle
        spent, passes = 0.0, 0
        while spent < min(5.0, args.cpu_seconds) and passes < 20:
            t0 = time.perf_counter()
            oracle.cache_append(p0.kv_new, p0.base.kv_cache, p0.base.block_table,
                                p0.base.cache_seqlens)
            oracle.q_absorb(p0.q_nope, p0.w_uk)
            spent += time.perf_counter() - t0
            passes += 1
        result["cpu_baseline"] = {
            "value": round(nbytes * passes / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"the whole workload, {passes} pass(es), {spent:.1f} s, fp64 C oracle "
                      "(single-threaded; includes copying the cache it appends to)"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


ATTENTION_METRIC = "Dense attention forward TFLOP/s and % of GB300 dense-bf16 tensor peak (1 GPU)"


def run_attention(args):
    """mla_attention_fwd per step (MLA prefill in the MHA form); torch's
    scaled_dot_product_attention timed on the same tensors beside it."""
    torch, world, rank, dev = _single_gpu_setup()
    from mla_decode_attention_07_gb300 import libmla
    libmla.load()
    w = W.ATTENTION_WORKLOADS[args.workload]
    peaks, peak_src = load_peaks()
    ai = w.make()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16))).to(dev).view(
        torch.bfloat16)
    q, k, v = t(ai.q), t(ai.k), t(ai.v)
    out = torch.empty((w.batch, w.seqlen, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.batch, w.heads, w.seqlen), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def ours(i):
        libmla.mla_attention_fwd(q, k, v, out, lse, w.causal, ai.scale, stream)

    for i in range(max(3, args.warmup)):
        ours(i)
    torch.cuda.synchronize()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error during warm-up: {libmla.mla_strerror(rc)}")
    sampler = ClockSampler(physical_gpu_index(dev.index))
    sampler.start()
    t_end = time.perf_counter() + 1.0
    i = 0
    while time.perf_counter() < t_end:
        ours(i)
        i += 1
        torch.cuda.synchronize()
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    ms = aggregate_max(_timed_loop(torch, stream, ours, K), world)
    clocks = sampler.stop()
    rc = libmla.mla_check_device_error(stream)
    if rc != 0:
        raise RuntimeError(f"device error in timed region: {libmla.mla_strerror(rc)}")
    tf = w.flops() / (ms * 1e-3) / 1e12
    sdpa = None
    try:
        import torch.nn.functional as F
        qt, kt, vt = q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)

        def theirs(i):
            F.scaled_dot_product_attention(qt, kt, vt, is_causal=w.causal, scale=ai.scale)

        for i in range(3):
            theirs(i)
        ms_t = _timed_loop(torch, stream, theirs, max(3, K // 2))
        sdpa = {"value": round(w.flops() / (ms_t * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(ms_t, 4), "ratio": round(ms_t / ms, 4),
                "how": "torch.nn.functional.scaled_dot_product_attention on the same tensors "
                       "(its own backend choice)"}
    except Exception as ex:   # backend without this head-dim combination
        sdpa = {"unavailable": f"{type(ex).__name__}: {str(ex)[:160]}"}
    result = {
        "metric": ATTENTION_METRIC, "value": round(tf * world, 3), "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "heads": w.heads,
                   "d_qk": w.d_qk, "d_v": w.d_v, "causal": w.causal,
                   "l2": f"inputs {w.bytes() / 1e6:.0f} MB per call (> L2)",
                   "parallelism": "single GPU" if world == 1 else f"{world} replicas"},
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                     "traffic": None, "kernel": "mla_attention_kernel",
                     "flops_per_call": w.flops(), "peak_source": f"{peak_src}: bf16 burst"},
        "sdpa": sdpa,
        "gpu_launches": K,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        rng = np.random.default_rng(0)
        n = 64
        while True:   # grow the row sample until the oracle works for a few seconds
            rows = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.heads, n),
                             rng.integers(0, w.seqlen, n)], 1).astype(np.int32)
            t0 = time.perf_counter()
            oracle.attention_rows(ai, rows)
            dt = time.perf_counter() - t0
            if dt >= min(5.0, args.cpu_seconds) or n >= 1 << 16:
                break
            n *= 4
        keys = sum(int(r[2]) + 1 if w.causal else w.seqlen for r in rows)
        result["cpu_baseline"] = {"value": 2.0 * (w.d_qk + w.d_v) * keys / dt / 1e12,
                                  "unit": "TFLOP/s", "cores": oracle.default_threads(),
                                  "kind": "oracle",
                                  "sample": f"{n} sampled query rows, fp64 C oracle, {dt:.2f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.workload in W.ATTENTION_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm is timed on the decode workloads; this line "
                              "carries its own cpu_baseline and SDPA comparison"}), flush=True)
        else:
            run_attention(args)
        return
    if args.workload in W.GEMM_WORKLOADS or args.workload in W.PROLOGUE_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm is timed on the decode workloads; this line "
                              "carries its own cpu_baseline or cuBLAS comparison"}), flush=True)
        elif args.workload in W.GEMM_WORKLOADS:
            run_gemm(args)
        else:
            run_prologue(args)
        return
    if args.workload in W.SPARSE_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm is timed on the dense workloads; the sparse "
                              "line carries its own cpu_baseline"}), flush=True)
        else:
            run_sparse(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
