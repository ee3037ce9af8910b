#!/usr/bin/env python3
"""Benchmark: multi-LoRA shrink + expand throughput (tokens/s per LoRA layer).

One step is one pass of the whole hot path over one batch: the device
grouping of the batch's tokens by LoRA id (once per batch), then shrink and
expand for each of ``--layers`` independent LoRA layers (distinct x, A, B, u,
y per layer, so the step's inputs are larger than the 129 MB L2 and every
byte comes from HBM).  The step is captured once in a CUDA graph and
replayed, as a serving engine does.

value   = n * layers / step time * ranks  (tokens/s per LoRA layer, whole job)
e2e     = the same metric with the per-step inputs (mapping, n, x, y of every
          layer) copied from pinned host memory and y copied back each step
roofline: the algorithmic bytes of the kernel with the largest share of the
          layer's device time / its measured launch time
          against the measured HBM copy bandwidth

``--impl reference`` times the fp64 CPU oracle instead (the only reference
this method has here), on the host cores, one bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gathered_rank_gemm_gb300 import workloads as W  # noqa: E402

METRIC = "LoRA shrink+expand tokens/s per layer; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {"expand": "gathered_rank_gemm_gb300/csrc/expand.cu",
                  "shrink": "gathered_rank_gemm_gb300/csrc/shrink.cu",
                  "expand-split": "gathered_rank_gemm_gb300/csrc/expand.cu",
                  "shrink-split": "gathered_rank_gemm_gb300/csrc/shrink.cu",
                  "shrink_expand": "gathered_rank_gemm_gb300/csrc/fused.cu",
                  "metadata": "gathered_rank_gemm_gb300/csrc/metadata.cu"}


# ---------------------------------------------------------------- accounting

def algorithmic_bytes(shape: W.LayerShape, mapping: np.ndarray):
    """Bytes the method must move per layer (not the dense work it skips)."""
    n, L, R, S, H = shape.num_tokens, shape.max_loras, shape.rank, shape.num_slices, shape.hidden
    m = mapping[:n]
    ids = m[(m >= 0) & (m < L)]
    n_l = int(ids.size)
    l_act = int(np.unique(ids).size)
    N = shape.out_width
    shrink = 2 * n_l * H + 2 * S * l_act * R * H + 4 * S * n_l * R
    expand = 4 * S * n_l * R + 2 * l_act * R * N + 4 * n_l * N
    meta = 4 * (2 * shape.max_num_tokens) + 4 * (2 * L + 3)
    flops = {"shrink": 2 * n_l * S * R * H, "expand": 2 * n_l * R * N}
    return dict(n_lora_tokens=n_l, active_loras=l_act, shrink=shrink, expand=expand,
                metadata=meta, flops=flops)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in (KERNEL_SOURCES[kernel], "gathered_rank_gemm_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[f"{kernel}/{workload}"]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        self.proc = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
        self.gpu = vis[local_rank] if local_rank < len(vis) and vis[local_rank].isdigit() \
            else local_rank
        self.tmp = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=self.tmp, stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().splitlines() if r.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        ids = {r[0].strip() for r in rows if r}
        target = str(self.gpu) if str(self.gpu) in ids else (sorted(ids)[0] if ids else "0")
        for r in rows:
            try:
                if r[0].strip() != target:
                    continue
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle timing

def oracle_sample_step(wl: W.Workload, max_tokens: int, threads: int, f16: bool = False):
    """One oracle pass (grouping + shrink + expand) over the first max_tokens
    adapter tokens of layer 0 (fp16 input words when f16); returns (tokens
    processed, seconds)."""
    import oracle
    sh, lay = wl.shape, wl.layers[0]
    n, L = sh.num_tokens, sh.max_loras
    m = wl.mapping.copy()
    if max_tokens < n:
        cut = n if max_tokens >= n else max_tokens
        m_sample = m.copy()
        m_sample[cut:n] = -1
    else:
        cut, m_sample = n, m
    t0 = time.perf_counter()
    oracle.prepare_metadata(m, n, L)
    u = oracle.shrink(lay.x, lay.lora_a, sh.scale, m_sample, n, L,
                      u_init=np.zeros((sh.num_slices, sh.max_num_tokens, sh.rank)),
                      num_threads=threads, f16=f16)
    oracle.expand(u, lay.lora_b, lay.y, m_sample, n, L, num_threads=threads, f16=f16)
    return cut, time.perf_counter() - t0


def oracle_sample_size(wl: W.Workload, budget_s: float, threads: int, f16: bool = False):
    n = wl.shape.num_tokens
    k = min(n, 32)
    _, dt = oracle_sample_step(wl, k, threads, f16)
    per_tok = dt / max(k, 1)
    return max(1, min(n, int(budget_s / max(per_tok, 1e-9))))


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl: W.Workload, seconds: float = 10.0, f16: bool = False):
    import oracle
    threads = oracle.max_threads()
    k = oracle_sample_size(wl, 2.0, threads, f16)
    tok, el, reps = 0, 0.0, 0
    while el < seconds and reps < 1000:
        t, dt = oracle_sample_step(wl, k, threads, f16)
        tok += t
        el += dt
        reps += 1
    # one thread, for about a quarter of the time (its own sample size)
    k1 = oracle_sample_size(wl, min(2.0, seconds / 4), 1, f16)
    tok1, el1 = 0, 0.0
    while el1 < seconds / 4 or tok1 == 0:
        t, dt = oracle_sample_step(wl, k1, 1, f16)
        tok1 += t
        el1 += dt
    return {"value": tok / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "single_thread_value": tok1 / el1, "cpu": cpu_model(),
            "sample": f"{reps} passes over the first {k} of {wl.shape.num_tokens} tokens of one "
                      f"{wl.shape.name} layer (grouping + shrink + expand, fp64), {el:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    shape = W.CONFIGS[args.config]
    wl = W.make_workload(shape, num_layers=1, seed=1000 + shape.index + 7919 * rank)
    f16 = args.dtype == "f16"
    if f16:
        wl.layers = [W.layer_as_f16(l) for l in wl.layers]
    threads = oracle.max_threads()
    k = oracle_sample_size(wl, 1.0, threads, f16)
    for _ in range(args.warmup):
        oracle_sample_step(wl, k, threads, f16)
    tok, el = 0, 0.0
    for _ in range(args.steps):
        t, dt = oracle_sample_step(wl, k, threads, f16)
        tok += t
        el += dt
    value = tok / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": shape.name, "max_num_tokens": shape.max_num_tokens,
                       "num_tokens": shape.num_tokens, "hidden": shape.hidden,
                       "slice_widths": list(shape.slice_widths), "max_loras": shape.max_loras,
                       "rank": shape.rank, "inputs": args.dtype},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"first {k} of {shape.num_tokens} tokens per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args, world, rank, local):
    import torch

    from gathered_rank_gemm_gb300 import binding
    from gathered_rank_gemm_gb300 import build as B

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    B.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = W.CONFIGS[args.config]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_layer = (shape.max_num_tokens * (shape.hidden + shape.out_width) * 2
                 + sum(shape.max_loras * shape.rank * (shape.hidden + w) * 2
                       for w in shape.slice_widths)
                 + 4 * shape.num_slices * shape.max_num_tokens * shape.rank)
    layers = args.layers or max(1, math.ceil(2 * l2 / per_layer))
    seed = 1000 + shape.index + 7919 * rank
    wl = W.make_workload(shape, num_layers=layers, seed=seed)
    T, L, n = shape.max_num_tokens, shape.max_loras, shape.num_tokens
    f16 = args.dtype == "f16"
    if f16:
        if args.paged:
            print(json.dumps({"error": "paged weights are bf16 only"}))
            return 1
        # the same draws rounded to fp16; the *_f16 entry points run them
        wl.layers = [W.layer_as_f16(l) for l in wl.layers]
    dt16 = torch.float16 if f16 else torch.bfloat16

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt16)

    stream = torch.cuda.Stream(dev)
    # the larger workspace lets lora_shrink_expand take its split-K path (stacked
    # weights only: the split-K halves have no paged form, so paged runs time
    # the cluster-path kernels their one call runs)
    ws_bytes = (None if args.paged else
                binding.lora_shrink_expand_workspace_size(T, L, shape.hidden, shape.slice_widths,
                                                          shape.rank))
    meta = binding.LoraMetadata(T, L, dev, workspace_bytes=ws_bytes)
    mapping = torch.from_numpy(wl.mapping).to(dev)
    n_dev = torch.tensor([n], dtype=torch.int32, device=dev)
    xs = [bf16(l.x) for l in wl.layers]
    ys = [bf16(l.y) for l in wl.layers]
    if args.paged:
        # every adapter's A_s[l] / B_s[l] in its own allocation, found through
        # one address table per layer and slice
        pages = []
        A_tab, B_tab = [], []
        for l in wl.layers:
            ta, tb = [], []
            for s_ in range(shape.num_slices):
                pa = [bf16(l.lora_a[s_][a]) for a in range(L)]
                pb = [bf16(l.lora_b[s_][a]) for a in range(L)]
                pages += pa + pb
                ta.append(torch.tensor([t.data_ptr() for t in pa], dtype=torch.int64, device=dev))
                tb.append(torch.tensor([t.data_ptr() for t in pb], dtype=torch.int64, device=dev))
            A_tab.append(ta)
            B_tab.append(tb)
    else:
        As = [[bf16(a) for a in l.lora_a] for l in wl.layers]
        Bs = [[bf16(b) for b in l.lora_b] for l in wl.layers]
    scales = None
    if args.lora_scales:
        scales = torch.from_numpy(np.random.default_rng(seed + 1).uniform(0.5, 1.5, L)
                                  .astype(np.float32)).to(dev)
    us = [torch.zeros(shape.num_slices, T, shape.rank, dtype=torch.float32, device=dev)
          for _ in wl.layers]
    torch.cuda.synchronize()

    # per layer, one lora_shrink_expand call: one fused kernel when the batch
    # fits on chip, else the shrink and expand kernels back to back
    per_layer_kernels = (2 if args.paged else
                         binding.lora_shrink_expand_kernels(T, L, shape.hidden,
                                                            shape.slice_widths, shape.rank))

    # which kernels lora_shrink_expand runs here: the split-K path leaves its
    # partial tiles behind the metadata part of the (zero-initialised) workspace
    split_k = False

    def step(which="all"):
        if which in ("all", "metadata", "profile"):
            meta.prepare(mapping, n_dev, stream)
        for k in range(layers):
            if which in ("all", "one_call", "profile"):
                if args.paged:
                    meta.shrink_expand_paged(xs[k], A_tab[k], B_tab[k], shape.slice_widths,
                                             shape.scale, us[k], ys[k], stream, scales)
                else:
                    meta.shrink_expand(xs[k], As[k], Bs[k], shape.scale, us[k], ys[k], stream,
                                       scales)
            # the kernels of the one call, timed one launch at a time
            if which == "shrink":
                if args.paged:
                    meta.shrink_paged(xs[k], A_tab[k], shape.rank, shape.scale, us[k], stream,
                                      scales)
                elif split_k:
                    meta.shrink_partials(xs[k], As[k], stream)
                else:
                    meta.shrink(xs[k], As[k], shape.scale, us[k], stream, scales)
            if which == "expand":
                if args.paged:
                    meta.expand_paged(us[k], B_tab[k], shape.slice_widths, ys[k], stream)
                elif split_k:
                    meta.expand_partials(shape.hidden, Bs[k], shape.scale, us[k], ys[k], stream,
                                         scales)
                else:
                    meta.expand(us[k], Bs[k], ys[k], stream)

    graphs = {}
    with torch.cuda.stream(stream):
        step()  # first call per device sets kernel attributes outside capture
    stream.synchronize()
    ws_base = binding.lora_workspace_size(T, L)
    split_k = (per_layer_kernels == 2 and meta.workspace.numel() > ws_base and
               bool(meta.workspace[ws_base:].any().item()))
    if args.mode == "profile":
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                step()
        stream.synchronize()
        if rank == 0:
            print(json.dumps({"mode": "profile", "workload": shape.name, "layers": layers,
                              "steps": args.steps, "launches": (1 + 2 * layers) * (args.steps + 1)}))
        return 0
    for which in ("all", "metadata", "one_call", "shrink", "expand"):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(which)
        graphs[which] = g

    def time_graph(g, reps, warm):
        with torch.cuda.stream(stream):
            for _ in range(warm):
                g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps  # ms per replay

    # ---- timed region: K steps, barrier + synchronize on both sides
    for _ in range(max(args.warmup, 3)):
        with torch.cuda.stream(stream):
            graphs["all"].replay()
    stream.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graphs["all"].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_step = e0.elapsed_time(e1) / args.steps
    # per-kernel launch times (each graph launches that kernel `layers` times)
    ms_meta = time_graph(graphs["metadata"], args.steps, 3)
    ms_one = time_graph(graphs["one_call"], args.steps, 3) / layers
    ms_shrink = time_graph(graphs["shrink"], args.steps, 3) / layers
    ms_expand = time_graph(graphs["expand"], args.steps, 3) / layers
    clk = clocks.stop()
    ms_step_max = max_over_ranks(ms_step, world, dev)

    # ---- end to end through the public API with host buffers
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_map = pin(wl.mapping)
    h_n = pin(np.array([n], np.int32))
    h_x = [pin(l.x.view(np.int16)) for l in wl.layers]
    h_y = [pin(l.y.view(np.int16)) for l in wl.layers]
    h_out = [torch.empty_like(h) .pin_memory() for h in h_y]
    h2d = h_map.numel() * 4 + 4 + sum(h.numel() * 2 for h in h_x) + sum(h.numel() * 2 for h in h_y)
    d2h = sum(h.numel() * 2 for h in h_y)

    def e2e_step():
        with torch.cuda.stream(stream):
            mapping.copy_(h_map, non_blocking=True)
            n_dev.copy_(h_n, non_blocking=True)
            for k in range(layers):
                xs[k].view(torch.int16).copy_(h_x[k], non_blocking=True)
                ys[k].view(torch.int16).copy_(h_y[k], non_blocking=True)
            graphs["all"].replay()
            for k in range(layers):
                h_out[k].copy_(ys[k].view(torch.int16), non_blocking=True)

    for _ in range(2):
        e2e_step()
    stream.synchronize()
    barrier(world)
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    stream.synchronize()
    ms_e2e = 1e3 * (time.perf_counter() - t0) / e2e_steps
    barrier(world)
    ms_e2e = max_over_ranks(ms_e2e, world, dev)

    alg = algorithmic_bytes(shape, wl.mapping)
    peak, peak_kind = load_peaks()
    if per_layer_kernels == 1:
        # one fused kernel per layer: it moves the bytes of both steps
        dominant, kernel_name = "shrink_expand", "lora_fused_kernel"
        dom_bytes, t_dom = alg["shrink"] + alg["expand"], ms_one
    else:
        # the kernel that takes the larger share of the layer's device time
        dominant = "expand" if ms_expand >= ms_shrink else "shrink"
        kernel_name = (f"lora_{dominant}_kernel" + (" (split-K)" if split_k else "")
                       + (" (paged weights)" if args.paged else ""))
        dom_bytes = alg[dominant]
        t_dom = ms_expand if dominant == "expand" else ms_shrink
    achieved = dom_bytes / (t_dom * 1e-3) / 1e9
    value = n * layers * world / (ms_step_max * 1e-3)
    e2e_value = n * layers * world / (ms_e2e * 1e-3)
    launches = (1 + per_layer_kernels * layers) * args.steps

    result = None
    if rank == 0:
        cpu = cpu_baseline(wl, seconds=args.cpu_seconds, f16=f16) if world == 1 else None
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": shape.name, "max_num_tokens": T, "num_tokens": n,
                       "hidden": shape.hidden, "slice_widths": list(shape.slice_widths),
                       "max_loras": L, "rank": shape.rank, "layers_per_step": layers,
                       "l2": f"inputs larger than L2: {layers} distinct layers, "
                             f"{layers * per_layer / 1e6:.0f} MB per step vs {l2 / 1e6:.0f} MB L2",
                       "graph": "one CUDA graph per step: grouping, then one lora_shrink_expand call per layer",
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "weights": "paged" if args.paged else "stacked",
                       "lora_scales": bool(args.lora_scales)},
            "roofline": {"bound": "hbm", "kernel": kernel_name,
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "frac_of_nominal_8tbs": achieved / 8000.0,
                         "algorithmic_bytes_per_launch": dom_bytes,
                         "traffic": recorded_traffic(dominant + ("-split" if split_k else "")
                                                     + ("-paged" if args.paged else ""),
                                                     shape.name)},
            "kernels_per_layer": per_layer_kernels,
            "one_call_path": "fused" if per_layer_kernels == 1 else ("split-K" if split_k else "cluster"),
            "kernels_us": {"metadata": 1e3 * ms_meta, "shrink_expand_one_call": 1e3 * ms_one,
                           "shrink": 1e3 * ms_shrink, "expand": 1e3 * ms_expand,
                           "layer_in_graph": 1e3 * ms_step / layers},
            "hbm_gbs": {"shrink": alg["shrink"] / (ms_shrink * 1e-3) / 1e9,
                        "expand": alg["expand"] / (ms_expand * 1e-3) / 1e9,
                        "shrink_expand_one_call": (alg["shrink"] + alg["expand"]) / (ms_one * 1e-3) / 1e9,
                        "layer": (alg["shrink"] + alg["expand"]) / (ms_step / layers * 1e-3) / 1e9},
            "tflops": {"shrink": alg["flops"]["shrink"] / (ms_shrink * 1e-3) / 1e12,
                       "expand": alg["flops"]["expand"] / (ms_expand * 1e-3) / 1e12},
            "lora_tokens": alg["n_lora_tokens"], "active_loras": alg["active_loras"],
            "lora_tokens_per_s": alg["n_lora_tokens"] * layers * world / (ms_step_max * 1e-3),
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(result), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(W.CONFIGS), default="decode_qkv")
    ap.add_argument("--layers", type=int, default=0, help="layers per step (0: >= 2x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--paged", action="store_true",
                    help="adapter weights as per-adapter pages found through address tables")
    ap.add_argument("--lora-scales", action="store_true", help="per-adapter scale factors")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="type of x, A, B and y (fp32 accumulation either way)")
    ap.add_argument("--mode", choices=["bench", "profile"], default="bench",
                    help="profile: only run --steps eager steps (for ncu launch lists)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 0)
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
