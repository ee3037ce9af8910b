#!/usr/bin/env python3
"""Benchmark: multi-LoRA shrink + expand throughput (tokens/s per LoRA layer).

A step is one pass of the whole hot path over one batch: the device grouping
of the batch's tokens by LoRA id (once per batch), then one
``lora_shrink_expand`` call (shrink + expand) for each of ``layers`` LoRA
layers held in distinct device buffers (so the step's inputs are larger than
twice the L2 and every byte comes from HBM).  Grouping and layers are
captured once as CUDA graphs and replayed, as a serving engine does.

With no ``--config`` every one of the five workloads is measured and the
JSON line's headline is ``down_proj_graph``, the largest one; the others are
in ``per_workload``.  For each workload:

value   = n * layers / t_layers  (tokens/s per LoRA layer, whole job): t_layers
          is the device time of the shrink + expand calls of a step, read with
          CUDA events around them; the grouping's time is reported on its own
          (``us.metadata_in_step``: inside the step, with the replay of its own
          graph; ``us.metadata_alone``: per kernel, from a graph of 16 grouping
          launches, the way the shrink and expand are timed alone) and
          ``value_with_metadata`` counts it in
ms_per_step = grouping + layers, device time of one step
e2e     = the same metric through the C ABI with each step's inputs (mapping,
          n, every layer's x and y) copied from pinned host memory and every
          layer's y copied back, host clock around the steps
roofline: the algorithmic bytes of the kernel with the largest share of the
          layer's device time / its launch time, against the measured HBM copy
          bandwidth; ``shrink_expand_frac`` is the same for the whole layer

The timed region is exactly --steps steps, bracketed by a barrier and a
device synchronisation; it is repeated until a workload has been timed for at
least --min-timed-ms, and ms_per_step is the median over the repetitions.
GPU clocks are sampled with nvidia-smi throughout.

``--impl reference`` times the fp64 CPU oracle instead (the only reference
this method has), on the host cores, one bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import shutil
import socket
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gathered_rank_gemm_gb300 import workloads as W  # noqa: E402

METRIC = "LoRA shrink+expand tokens/s per layer; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
HEADLINE = "down_proj_graph"
ORDER = ("tiny", "decode_qkv", "chunked_prefill", "mlp_gate_up", "down_proj_graph")
FALLBACK_HBM_GBS = 6800.0
# the sources of each timed kernel (the expand of rank 128 on large batches is
# the tcgen05 kernel)
KERNEL_SOURCES = {"expand": ("gathered_rank_gemm_gb300/csrc/expand.cu",
                             "gathered_rank_gemm_gb300/csrc/expand_tc.cu"),
                  "shrink": ("gathered_rank_gemm_gb300/csrc/shrink.cu",),
                  "expand-split": ("gathered_rank_gemm_gb300/csrc/expand.cu",),
                  "shrink-split": ("gathered_rank_gemm_gb300/csrc/shrink.cu",),
                  "shrink_expand": ("gathered_rank_gemm_gb300/csrc/fused.cu",),
                  "metadata": ("gathered_rank_gemm_gb300/csrc/metadata.cu",)}


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


def layer_bytes(shape: W.LayerShape) -> int:
    """Device bytes of one layer's buffers (x, y, u, A, B)."""
    return (shape.max_num_tokens * (shape.hidden + shape.out_width) * 2
            + sum(shape.max_loras * shape.rank * (shape.hidden + w) * 2 for w in shape.slice_widths)
            + 4 * shape.num_slices * shape.max_num_tokens * shape.rank)


def layers_per_step(shape: W.LayerShape, l2_bytes: int) -> int:
    """Distinct layer buffers per step: together more than twice the L2, and
    at least four, so a layer's inputs were evicted before it comes round."""
    return max(4, math.ceil(2 * l2_bytes / layer_bytes(shape)))


def config_of(shape: W.LayerShape, args, l2_bytes: int, world: int) -> dict:
    """The workload and how it is run (the same for both arms)."""
    layers = args.layers or layers_per_step(shape, l2_bytes)
    return {"workload": shape.name, "max_num_tokens": shape.max_num_tokens,
            "num_tokens": shape.num_tokens, "hidden": shape.hidden,
            "slice_widths": list(shape.slice_widths), "max_loras": shape.max_loras,
            "rank": shape.rank, "inputs": args.dtype,
            "weights": "paged" if args.paged else "stacked",
            "lora_scales": bool(args.lora_scales), "layers_per_step": layers,
            "l2": f"inputs larger than L2: {layers} distinct layer buffers, "
                  f"{layers * layer_bytes(shape) / 1e6:.0f} MB per step vs "
                  f"{l2_bytes / 1e6:.0f} MB L2",
            "graph": "per step: one CUDA graph of the grouping, one of the "
                     "lora_shrink_expand calls of every layer",
            "parallelism": f"replicas x{world} (independent batches, no collective)"}


def device_l2_bytes() -> int:
    """L2 size of the GPU (GB300: about 130 MB when none is visible)."""
    try:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except Exception:
        pass
    return 132_120_576


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
    for rel in KERNEL_SOURCES[kernel] + ("gathered_rank_gemm_gb300/csrc/common.cuh",):
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
    """nvidia-smi clock / throttle samples, each stamped with the host clock."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_rank: int):
        self.proc = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
        self.gpu = vis[local_rank] if local_rank < len(vis) and vis[local_rank].isdigit() \
            else str(local_rank)
        self.rows = []
        self.reader = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

        def read():
            for line in self.proc.stdout:
                if line.strip():
                    self.rows.append((time.time(), [c.strip() for c in line.split(",")]))
        self.reader = threading.Thread(target=read, daemon=True)
        self.reader.start()
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)

    def summary(self, windows=None):
        """Median SM clock, max clock and active throttle reasons over the
        samples inside the host-time windows (all samples when None)."""
        ids = {r[0] for _, r in self.rows if r}
        target = self.gpu if self.gpu in ids else (sorted(ids)[0] if ids else "0")
        sm, mx, reasons = [], [], set()
        for ts, r in self.rows:
            if windows is not None and not any(a <= ts <= b for a, b in windows):
                continue
            try:
                if r[0] != target:
                    continue
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, val in zip(self.REASONS, r[5:9]):
                    if val.lower() == "active":
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
    tokens of layer 0 (fp16 input words when f16); returns (tokens processed,
    seconds)."""
    import oracle
    sh, lay = wl.shape, wl.layers[0]
    n, L = sh.num_tokens, sh.max_loras
    m = wl.mapping.copy()
    cut = min(max_tokens, n)
    m_sample = m.copy()
    m_sample[cut:n] = -1
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
    """The oracle on all host cores (and, for a quarter of the time, on one)."""
    import oracle
    threads = oracle.max_threads()
    k = oracle_sample_size(wl, min(2.0, seconds / 2), threads, f16)
    tok, el, reps = 0, 0.0, 0
    while el < seconds and reps < 1000:
        t, dt = oracle_sample_step(wl, k, threads, f16)
        tok += t
        el += dt
        reps += 1
    k1 = oracle_sample_size(wl, min(1.0, seconds / 8), 1, f16)
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
    """The oracle as the reference arm: rank 0 alone runs and prints."""
    if rank != 0:
        return 0
    import oracle
    shape = W.CONFIGS[args.config if args.config != "all" else HEADLINE]
    wl = W.make_workload(shape, num_layers=1, seed=1000 + shape.index)
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
            "config": config_of(shape, args, device_l2_bytes(), world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"first {k} of {shape.num_tokens} tokens per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

class WorkloadRun:
    """One workload on the device: buffers, graphs and timings."""

    def __init__(self, args, shape, dev, stream, rank, l2):
        import torch

        from gathered_rank_gemm_gb300 import binding
        self.torch, self.binding = torch, binding
        self.args, self.shape, self.dev, self.stream = args, shape, dev, stream
        self.l2 = l2
        self.layers = args.layers or layers_per_step(shape, l2)
        self.seed = 1000 + shape.index + 7919 * rank
        # one layer's values drawn on the host, held in `layers` distinct
        # device buffers (distinct addresses are what the L2 sees)
        wl = W.make_workload(shape, num_layers=1, seed=self.seed)
        self.f16 = args.dtype == "f16"
        if self.f16:
            wl.layers = [W.layer_as_f16(l) for l in wl.layers]
        self.wl = wl
        T, L, n = shape.max_num_tokens, shape.max_loras, shape.num_tokens
        dt16 = torch.float16 if self.f16 else torch.bfloat16
        lay = wl.layers[0]

        def dev16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(dt16)

        # the larger workspace lets lora_shrink_expand take its split-K path
        # (stacked weights only: the split-K halves have no paged form)
        ws_bytes = (None if args.paged else
                    binding.lora_shrink_expand_workspace_size(T, L, shape.hidden,
                                                              shape.slice_widths, shape.rank))
        self.meta = binding.LoraMetadata(T, L, dev, workspace_bytes=ws_bytes)
        self.mapping = torch.from_numpy(wl.mapping).to(dev)
        self.n_dev = torch.tensor([n], dtype=torch.int32, device=dev)
        x0, y0 = dev16(lay.x), dev16(lay.y)
        self.xs = [x0] + [x0.clone() for _ in range(self.layers - 1)]
        self.ys = [y0] + [y0.clone() for _ in range(self.layers - 1)]
        a0 = [dev16(a) for a in lay.lora_a]
        b0 = [dev16(b) for b in lay.lora_b]
        self.As = [a0] + [[a.clone() for a in a0] for _ in range(self.layers - 1)]
        self.Bs = [b0] + [[b.clone() for b in b0] for _ in range(self.layers - 1)]
        if args.paged:
            # every adapter's A_s[l] / B_s[l] viewed as its own page, found
            # through one address table per layer and slice
            self.A_tab = [[torch.tensor([a[l].data_ptr() for l in range(L)], dtype=torch.int64,
                                        device=dev) for a in As] for As in self.As]
            self.B_tab = [[torch.tensor([b[l].data_ptr() for l in range(L)], dtype=torch.int64,
                                        device=dev) for b in Bs] for Bs in self.Bs]
        self.scales = None
        if args.lora_scales:
            self.scales = torch.from_numpy(np.random.default_rng(self.seed + 1).uniform(0.5, 1.5, L)
                                           .astype(np.float32)).to(dev)
        self.us = [torch.zeros(shape.num_slices, T, shape.rank, dtype=torch.float32, device=dev)
                   for _ in range(self.layers)]
        torch.cuda.synchronize()
        # the path one lora_shrink_expand call takes here (fused kernel, split-K
        # pair or cluster pair)
        self.path = binding.lora_shrink_expand_path(T, L, shape.hidden, shape.slice_widths,
                                                    shape.rank, self.meta.workspace.numel(),
                                                    fp16=self.f16, paged=args.paged)
        self.per_layer_kernels = 1 if self.path == binding.LORA_PATH_FUSED else 2
        self.split_k = self.path == binding.LORA_PATH_SPLIT_PAIR
        self.graphs = {}

    def launch(self, which):
        """Enqueue one step's part: metadata, layers (one call each), or the
        shrink / expand alone (lora_shrink / lora_expand, or the split-K pair's
        halves where the one call takes that path; one launch per layer)."""
        m, sh, s = self.meta, self.shape, self.stream
        if which == "metadata":
            m.prepare(self.mapping, self.n_dev, s)
            return
        if which == "metadata_x16":
            for _ in range(16):
                m.prepare(self.mapping, self.n_dev, s)
            return
        for k in range(self.layers):
            if which == "layers":
                if self.args.paged:
                    m.shrink_expand_paged(self.xs[k], self.A_tab[k], self.B_tab[k],
                                          sh.slice_widths, sh.scale, self.us[k], self.ys[k], s,
                                          self.scales)
                else:
                    m.shrink_expand(self.xs[k], self.As[k], self.Bs[k], sh.scale, self.us[k],
                                    self.ys[k], s, self.scales)
            elif which == "shrink":
                if self.args.paged:
                    m.shrink_paged(self.xs[k], self.A_tab[k], sh.rank, sh.scale, self.us[k], s,
                                   self.scales)
                elif self.split_k:
                    m.shrink_partials(self.xs[k], self.As[k], s)
                else:
                    m.shrink(self.xs[k], self.As[k], sh.scale, self.us[k], s, self.scales)
            elif which == "expand":
                if self.args.paged:
                    m.expand_paged(self.us[k], self.B_tab[k], sh.slice_widths, self.ys[k], s)
                elif self.split_k:
                    m.expand_partials(sh.hidden, self.Bs[k], sh.scale, self.us[k], self.ys[k], s,
                                      self.scales)
                else:
                    m.expand(self.us[k], self.Bs[k], self.ys[k], s)

    def capture(self):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.launch("metadata")   # first calls per device set kernel attributes
            self.launch("layers")     # outside any capture
        self.stream.synchronize()
        base = self.binding.lora_workspace_size(self.shape.max_num_tokens, self.shape.max_loras)
        if self.split_k:
            # the split paths leave partial tiles behind the metadata part of
            # the (zero-initialised) workspace: check that this one ran
            assert bool(self.meta.workspace[base:].any().item()), "split-K path did not run"
        for which in ("metadata", "metadata_x16", "layers", "shrink", "expand"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.launch(which)
            self.graphs[which] = g

    def time_graph(self, which, min_ms=50.0):
        """Device ms per replay of one graph (CUDA events on the stream)."""
        torch, g = self.torch, self.graphs[which]
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                g.replay()
        self.stream.synchronize()
        reps, total = 0, 0.0
        while total < min_ms or reps < 10:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            with torch.cuda.stream(self.stream):
                for _ in range(10):
                    g.replay()
            e1.record(self.stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
            reps += 10
        return total / reps

    def timed_steps(self, steps, world):
        """Exactly `steps` steps, barrier + synchronize on both sides; returns
        (ms per step, ms of the layers per step, ms of the grouping per step,
        host window)."""
        torch = self.torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        h0 = time.time()
        with torch.cuda.stream(self.stream):
            for e in ev:
                e[0].record(self.stream)
                self.graphs["metadata"].replay()
                e[1].record(self.stream)
                self.graphs["layers"].replay()
                e[2].record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        h1 = time.time()
        meta = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
        lay = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
        step = sum(e[0].elapsed_time(e[2]) for e in ev) / steps
        return step, lay, meta, (h0, h1)

    def measure(self, steps, warmup, min_ms, world):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for _ in range(max(warmup, 3)):
                self.graphs["metadata"].replay()
                self.graphs["layers"].replay()
        self.stream.synchronize()
        reps, windows = [], []
        spent = 0.0
        while spent < min_ms or not reps:
            step, lay, meta, win = self.timed_steps(steps, world)
            reps.append((step, lay, meta))
            windows.append(win)
            spent += step * steps
        self.windows = windows
        self.reps = reps
        med = sorted(reps, key=lambda r: r[0])[len(reps) // 2]
        self.ms_step, self.ms_layers, self.ms_meta = med
        self.timed_ms = spent
        # each kernel of the layer on its own (graphs of `layers` launches)
        self.ms_one = self.time_graph("layers") / self.layers
        self.ms_shrink = self.time_graph("shrink") / self.layers
        self.ms_expand = self.time_graph("expand") / self.layers
        self.ms_meta_alone = self.time_graph("metadata_x16") / 16

    def e2e(self, steps, world):
        """Steps through the public API with host buffers: the step's inputs
        copied from pinned host memory and every layer's y copied back."""
        torch = self.torch
        lay = self.wl.layers[0]
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        h_map = pin(self.wl.mapping)
        h_n = pin(np.array([self.shape.num_tokens], np.int32))
        h_x = pin(lay.x.view(np.int16))
        h_y = pin(lay.y.view(np.int16))
        h_out = [torch.empty_like(h_y).pin_memory() for _ in range(self.layers)]
        h2d = h_map.numel() * 4 + 4 + self.layers * (h_x.numel() * 2 + h_y.numel() * 2)
        d2h = self.layers * h_y.numel() * 2

        def one():
            with torch.cuda.stream(self.stream):
                self.mapping.copy_(h_map, non_blocking=True)
                self.n_dev.copy_(h_n, non_blocking=True)
                for k in range(self.layers):
                    self.xs[k].view(torch.int16).copy_(h_x, non_blocking=True)
                    self.ys[k].view(torch.int16).copy_(h_y, non_blocking=True)
                self.graphs["metadata"].replay()
                self.graphs["layers"].replay()
                for k in range(self.layers):
                    h_out[k].copy_(self.ys[k].view(torch.int16), non_blocking=True)

        for _ in range(2):
            one()
        self.stream.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        self.stream.synchronize()
        ms = 1e3 * (time.perf_counter() - t0) / steps
        barrier(world)
        return ms, h2d, d2h

    def record(self, peak, peak_kind, world, ms_layers_max, ms_step_max):
        sh = self.shape
        n, T, L = sh.num_tokens, sh.max_num_tokens, sh.max_loras
        alg = algorithmic_bytes(sh, self.wl.mapping)
        both = alg["shrink"] + alg["expand"]
        if self.per_layer_kernels == 1:
            # one fused kernel per layer: it moves the bytes of both steps
            dominant, kernel_name = "shrink_expand", "lora_fused_kernel"
            dom_bytes, t_dom = both, self.ms_one
        else:
            dominant = "expand" if self.ms_expand >= self.ms_shrink else "shrink"
            kernel_name = (f"lora_{dominant}_kernel" + (" (split-K)" if self.split_k else "")
                           + (" (paged weights)" if self.args.paged else ""))
            dom_bytes = alg[dominant]
            t_dom = self.ms_expand if dominant == "expand" else self.ms_shrink
        gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
        achieved = gbs(dom_bytes, t_dom)
        ms_layer = ms_layers_max / self.layers
        key = dominant + ("-split" if self.split_k else "") + ("-paged" if self.args.paged else "")
        return {
            "config": config_of(sh, self.args, self.l2, world),
            "layers_per_step": self.layers,
            "one_call_path": self.binding.PATH_NAMES[self.path],
            "kernels_per_layer": self.per_layer_kernels,
            "tokens_per_s": n * self.layers * world / (ms_layers_max * 1e-3),
            "tokens_per_s_with_metadata": n * self.layers * world / (ms_step_max * 1e-3),
            "lora_tokens_per_s": alg["n_lora_tokens"] * self.layers * world / (ms_layers_max * 1e-3),
            "lora_tokens": alg["n_lora_tokens"], "active_loras": alg["active_loras"],
            "us": {"layer_in_step": 1e3 * ms_layer, "metadata_in_step": 1e3 * self.ms_meta,
                   "metadata_alone": 1e3 * self.ms_meta_alone,
                   "one_call": 1e3 * self.ms_one, "shrink": 1e3 * self.ms_shrink,
                   "expand": 1e3 * self.ms_expand},
            "algorithmic_bytes": {"shrink": alg["shrink"], "expand": alg["expand"]},
            "hbm": {"peak_gbs": peak, "peak_source": peak_kind,
                    "shrink_expand_gbs": gbs(both, ms_layer),
                    "shrink_expand_frac": gbs(both, ms_layer) / peak,
                    "one_call_frac": gbs(both, self.ms_one) / peak,
                    "shrink_frac": gbs(alg["shrink"], self.ms_shrink) / peak,
                    "expand_frac": gbs(alg["expand"], self.ms_expand) / peak},
            "tflops": {"shrink": alg["flops"]["shrink"] / (self.ms_shrink * 1e-3) / 1e12,
                       "expand": alg["flops"]["expand"] / (self.ms_expand * 1e-3) / 1e12},
            "roofline": {"bound": "hbm", "kernel": kernel_name, "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": peak_kind, "frac_of_nominal_8tbs": achieved / 8000.0,
                         "algorithmic_bytes_per_launch": dom_bytes,
                         "traffic": recorded_traffic(key, sh.name)},
            "timed": {"steps_per_repeat": self.args.steps,
                      "repeats": len(self.reps), "ms": self.timed_ms,
                      "ms_per_step_repeats": [r[0] for r in self.reps]},
        }

    def free(self):
        self.graphs.clear()
        for name in ("xs", "ys", "As", "Bs", "us", "meta", "mapping", "n_dev"):
            setattr(self, name, None)


def run_ours(args, world, rank, local):
    import torch

    from gathered_rank_gemm_gb300 import binding
    from gathered_rank_gemm_gb300 import build as B

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device: the library has no CPU path"}))
        return 1
    if args.paged and args.dtype == "f16":
        print(json.dumps({"error": "paged weights are bf16 only"}))
        return 1
    B.build()
    binding.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    names = ORDER if args.config == "all" else (args.config,)
    headline = HEADLINE if args.config == "all" else args.config
    peak, peak_kind = load_peaks()
    stream = torch.cuda.Stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    records, head = {}, None
    if args.mode == "profile":
        # eager steps only (grouping + every layer's call), for profiler launch lists
        clocks.stop()
        run = WorkloadRun(args, W.CONFIGS[headline], dev, stream, rank, l2)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                run.launch("metadata")
                run.launch(args.profile_part)
        stream.synchronize()
        if rank == 0:
            print(json.dumps({"mode": "profile", "workload": headline, "layers": run.layers,
                              "steps": args.steps, "path": binding.PATH_NAMES[run.path]}))
        return 0
    try:
        for name in names:
            run = WorkloadRun(args, W.CONFIGS[name], dev, stream, rank, l2)
            run.capture()
            # the headline is timed longer, so the clock record has tens of samples
            min_ms = args.min_timed_ms * (5.0 if name == headline else 1.0)
            run.measure(args.steps, args.warmup, min_ms, world)
            ms_layers = max_over_ranks(run.ms_layers, world, dev)
            ms_step = max_over_ranks(run.ms_step, world, dev)
            rec = run.record(peak, peak_kind, world, ms_layers, ms_step)
            rec["clocks"] = clocks.summary(run.windows)
            if name == headline:
                ms_e2e, h2d, d2h = run.e2e(max(3, min(args.steps, 10)), world)
                ms_e2e = max_over_ranks(ms_e2e, world, dev)
                rec["e2e"] = {"value": run.shape.num_tokens * run.layers * world / (ms_e2e * 1e-3),
                              "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                              "ms_per_step": ms_e2e}
                head = (run, ms_layers, ms_step)
            rec["_wl"] = run.wl
            records[name] = rec
            run.free()
            torch.cuda.empty_cache()
    finally:
        clocks.stop()
    if rank != 0:
        return 0
    # the oracle on the host cores, a bounded sample of each workload
    for name, rec in records.items():
        wl = rec.pop("_wl")
        if world == 1:
            secs = args.cpu_seconds if name == headline else max(1.0, args.cpu_seconds / 4)
            rec["cpu_baseline"] = cpu_baseline(wl, seconds=secs, f16=args.dtype == "f16")
        else:
            rec["cpu_baseline"] = None
    run, ms_layers, ms_step = head
    h = records[headline]
    result = {
        "metric": METRIC, "value": h["tokens_per_s"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic",
        "config": h["config"],
        "value_with_metadata": h["tokens_per_s_with_metadata"],
        "ms_layers_per_step": ms_layers,
        "roofline": h["roofline"],
        "shrink_expand_frac": h["hbm"]["shrink_expand_frac"],
        "cpu_baseline": h["cpu_baseline"],
        "e2e": h.pop("e2e"),
        # this library's kernels in the headline's timed region: the grouping
        # and the kernels of every layer's call, per step
        "gpu_launches": h["timed"]["repeats"] * args.steps * (1 + h["kernels_per_layer"]
                                                              * h["layers_per_step"]),
        "timed": h["timed"],
        "clocks": h["clocks"],
        "clocks_all_workloads": clocks.summary(None),
        "per_workload": records,
    }
    print(json.dumps(result), flush=True)
    return 0


def _spawn_ranks(argv, n):
    """One process per GPU (rank = local rank), launched here when no
    launcher set WORLD_SIZE; returns the worst exit code."""
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(argv, r, n, port)) for r in range(n)]
    for p in procs:
        p.start()
    for p in procs:
        p.join()
    return max(abs(p.exitcode or 0) for p in procs)


def _rank_main(argv, rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.exit(main(argv))


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["all"] + list(W.CONFIGS), default="all",
                    help="one workload, or all five (headline: down_proj_graph)")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per step (0: at least 4 and more than 2x L2)")
    ap.add_argument("--min-timed-ms", type=float, default=200.0,
                    help="repeat the timed --steps steps until a workload was timed this long")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--paged", action="store_true",
                    help="adapter weights as per-adapter pages found through address tables")
    ap.add_argument("--lora-scales", action="store_true", help="per-adapter scale factors")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="type of x, A, B and y (fp32 accumulation either way)")
    ap.add_argument("--mode", choices=["bench", "profile"], default="bench",
                    help="profile: only run --steps eager steps of one workload (for ncu)")
    ap.add_argument("--profile-part", choices=["layers", "shrink", "expand"], default="layers",
                    help="profile mode: per layer the one call (layers), or lora_shrink / "
                         "lora_expand alone")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 0)
    return args


def main(argv=None):
    args = parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        if args.impl == "ours":
            import torch
            have = torch.cuda.device_count() if torch.cuda.is_available() else 0
            if have < args.gpus:
                print(json.dumps({"error": f"--gpus {args.gpus} needs {args.gpus} CUDA devices, "
                                           f"{have} visible"}), flush=True)
                return 1
        return _spawn_ranks(sys.argv[1:] if argv is None else list(argv), args.gpus)
    world, rank, local = dist_setup(args)
    if args.gpus != world:
        if rank == 0:
            print(json.dumps({"error": f"--gpus {args.gpus} but the launcher started {world} "
                                       "ranks"}), flush=True)
        return 1
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
