#!/usr/bin/env python3
"""Benchmark of the clip + AdamW optimizer step: parameters per second and achieved HBM bandwidth on one GB300.

One step = ClipGradNorms (norm partials + fixed-order finalize) and AdamWSteps over the whole parameter list, through
the C ABI's one-step entry point mica_clip_adamw_step (via the Python binding), inputs resident in HBM. Prints one
JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gpt2_small] [--impl mica|reference]

--impl reference times the CPU oracle (the plain single-threaded C step) on the host cores instead, on a bounded
sample of the same workload. Under torchrun with N > 1 every rank runs the whole step on its own GPU (each rank a
replica, as data-parallel training steps its replicated parameters); the time is the slowest rank's. With --shard
the ranks split the list instead (each steps its own part after one all-gather of the norm's square sums).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "clip+AdamW params/sec and achieved HBM GB/s (% of 8 TB/s roofline), 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRCS = [os.path.join(ROOT, "clip_tensor_adamw_gb300", "csrc", f)
               for f in ("adamw.cu", "adam.cuh", "stream.cuh", "plan.h")]
PROFILE = os.path.join(ROOT, "profiles", "adamw_gpt2_small.md")


# ----------------------------------------------------------------------------------------------------------------
# the byte model: algorithmic bytes per parameter
# ----------------------------------------------------------------------------------------------------------------

def adamw_bytes_per_param(wl: workloads.Workload, zero_grad: bool = False, opt: str = "adamw") -> float:
    """The update kernel. AdamW: w read + write (8), g read (4 or 2), m and v read + write (16 float32, 8 packed
    BF16): 28 B/param with float32 moments, 20 with packed ones. SGD: w (8) and g; with momentum also the buffer's
    read + write (8). The gradient's zero write (4 or 2) only with zero_grad."""
    g = 2.0 if wl.grad_dtype == "f16" else 4.0
    if opt == "sgd":
        mv = 0.0
    elif opt == "momentum":
        mv = 8.0
    else:
        mv = {"bf16x2": 8.0, "bf16x2_m": 12.0}.get(wl.moments, 16.0)
    return 8.0 + g + mv + (g if zero_grad else 0.0)


def step_bytes_per_param(wl: workloads.Workload, zero_grad: bool = False, opt: str = "adamw") -> float:
    """The whole step: the norm's read of g plus the update kernel (AdamW: 28 / 20 B + 4 B with float32
    gradients). With opt "accumulate" the norm is fused into the gradient's last write, g += a: that kernel reads
    g and a and writes g (12 B with float32 gradients), and the norm reads nothing more."""
    g = 2.0 if wl.grad_dtype == "f16" else 4.0
    if opt == "accumulate":
        return 3 * g + adamw_bytes_per_param(wl, zero_grad, "adamw")
    return g + adamw_bytes_per_param(wl, zero_grad, opt)


def describe(wl: workloads.Workload) -> str:
    return (f"{wl.name}: {len(wl.sizes)} tensors, {wl.params:,} params, {wl.grad_dtype} grads, "
            f"{'packed BF16' if wl.moments == 'bf16x2' else 'f32'} moments")


# ----------------------------------------------------------------------------------------------------------------
# peaks, profiles, clocks
# ----------------------------------------------------------------------------------------------------------------

def _hbm_gbs_in(d) -> float | None:
    """The HBM copy bandwidth in GB/s in a peaks record: the first number whose key path names HBM (or DRAM /
    memory) and a GB/s or TB/s unit, searched depth-first; a TB/s figure is converted."""
    found = []

    def walk(x, path):
        if isinstance(x, dict):
            for k, v in x.items():
                walk(v, path + [str(k).lower()])
        elif isinstance(x, (int, float)) and not isinstance(x, bool) and x > 0:
            key = "_".join(path)
            if any(m in key for m in ("hbm", "dram", "mem")) and "bf16" not in key and "tflop" not in key:
                if any(u in key for u in ("gbs", "gb_s", "gbps", "gb/s")):
                    found.append(float(x))
                elif any(u in key for u in ("tbs", "tb_s", "tbps", "tb/s")):
                    found.append(1e3 * float(x))
    walk(d, [])
    return found[0] if found else None


def hbm_peak(path: str | None = None) -> tuple[float, str]:
    """The measured HBM copy peak (GB/s) from MEASURED_PEAKS.json when present, else the fallback figure."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = _hbm_gbs_in(json.load(f))
        if v is not None and 100.0 < v < 100000.0:
            return v, "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha() -> str:
    """The first 16 hex digits of the SHA-256 of the AdamW kernel's sources (adamw.cu, adam.cuh, stream.cuh, plan.h)."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic() -> float | None:
    """DRAM bytes per AdamW launch from the committed ncu summary, if it was taken on the current kernel source."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    sha = kernel_source_sha()
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_b = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows: list[tuple[float, list[str]]] = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5.0:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for t, r in self.rows if t0 - 0.05 <= t <= t1 + 0.15]
        if not inside:  # a region shorter than the sampling period: the nearest sample after it began
            after = [r for t, r in self.rows if t >= t0]
            inside = after[:1] or [r for _, r in self.rows[-1:]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        mx = [num(r[2]) for r in inside if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------------------------------------------------------
# the CPU oracle: the reference arm and the cpu_baseline
# ----------------------------------------------------------------------------------------------------------------

def oracle_sample(wl: workloads.Workload, target_params: int):
    """A bounded sample of the workload for the oracle: its first tensors up to ~target_params parameters (at
    least one tensor), on the host."""
    sizes, tot = [], 0
    for n in wl.sizes:
        if sizes and tot + n > target_params:
            break
        sizes.append(n)
        tot += n
    st = workloads.make_state(wl, "cpu", sizes=sizes)
    workloads.fill_grad(st, 1)
    return workloads.host_lists(st), tot, len(sizes)


def time_oracle(wl: workloads.Workload, target_params: int, min_seconds: float, max_steps: int):
    import oracle
    ora = oracle.Oracle()
    host, params, ntens = oracle_sample(wl, target_params)
    hp = oracle.Hyper(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, step=1)
    times = []
    t_all = time.perf_counter()
    t = 0
    while t < max_steps and (time.perf_counter() - t_all < min_seconds or t == 0):
        t += 1
        t0 = time.perf_counter()
        ora.clip_adamw_step(*host, oracle.Hyper(**{**hp.__dict__, "step": t}), wl.max_norm, wl.inv_scale)
        times.append(time.perf_counter() - t0)
    return params, ntens, times


def host_cpu() -> dict:
    """The host the CPU baseline ran on: its architecture, CPU model (as /proc/cpuinfo names it) and thread count."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            fields = dict(line.split(":", 1) for line in f if ":" in line)
        fields = {k.strip(): v.strip() for k, v in fields.items()}
        model = fields.get("model name") or (
            f"implementer {fields.get('CPU implementer', '?')} part {fields.get('CPU part', '?')}")
    except OSError:
        pass
    return {"arch": platform.machine(), "cpu": model, "nproc": os.cpu_count()}


def run_config(wl: workloads.Workload, world: int) -> dict:
    """The `config` of both arms' JSON lines: the workload the metric is quoted on."""
    bpp = step_bytes_per_param(wl)
    return {"workload": describe(wl), "params": wl.params, "tensors": len(wl.sizes), "moments": wl.moments,
            "grad_dtype": wl.grad_dtype, "zero_grad": False, "bytes_per_param": bpp,
            "l2": f"inputs larger than L2 ({wl.params * bpp / 1e9:.2f} GB moved per step; no flush)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, wl: workloads.Workload) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    params, ntens, times = None, None, []
    import oracle
    ora = oracle.Oracle()
    host, params, ntens = oracle_sample(wl, max(1, wl.params // 8))
    hp0 = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay)
    for t in range(1, args.warmup + args.steps + 1):
        t0 = time.perf_counter()
        ora.clip_adamw_step(*host, oracle.Hyper(step=t, **hp0), wl.max_norm, wl.inv_scale)
        if t > args.warmup:
            times.append(time.perf_counter() - t0)
    sec = sum(times)
    value = params * len(times) / sec
    sample = f"first {ntens} of {len(wl.sizes)} tensors of {wl.name} ({params:,} of {wl.params:,} params) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": run_config(wl, args.gpus),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host_cpu()},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------------------------------
# the GPU step
# ----------------------------------------------------------------------------------------------------------------

def slowest_rank_ms(ms: float, dist, device) -> float:
    """The timed region of the slowest rank: every rank's time, reduced by MAX over the process group."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, params: int, steps: int, total_ms: float) -> float:
    """Parameters stepped per second by the whole job: every rank steps its own full list (weak scaling)."""
    return world * params * steps / (total_ms / 1e3)


def decay_groups(wl: workloads.Workload):
    """Parameter groups of a transformer's usual split: matrices decay (group 0); vectors do not and take half the
    lr (group 1)."""
    group = [0 if len(s) >= 2 else 1 for s in wl.shapes]
    return group, [dict(lr=wl.lr, weight_decay=wl.weight_decay), dict(lr=wl.lr / 2, weight_decay=0.0)]


SGD_LR, SGD_MOMENTUM = 0.1, 0.9

MIN_STEPS_EXTRA, MIN_MS_EXTRA = 200, 50.0


def extra_steps(est_ms_per_step: float) -> int:
    """Timed steps for a secondary workload: at least MIN_STEPS_EXTRA and at least MIN_MS_EXTRA of GPU time, so that
    short steps are not timed on a region of a few milliseconds."""
    return max(MIN_STEPS_EXTRA, math.ceil(MIN_MS_EXTRA / max(est_ms_per_step, 1e-4)))


def measure(wl: workloads.Workload, steps: int, warmup: int, zero_grad: bool, dist=None, sampler=None,
            coupled_l2: bool = False, opt: str = "adamw", per_kernel: bool = True):
    """Times `steps` steps of the whole hot path on the device (inputs resident): the norm and clip factor, then the
    update (``opt``: "adamw", "adamw_groups", "sgd" or "momentum"; "accumulate": each step first adds a second
    gradient contribution into g with the norm fused into that add, then AdamW). Returns a dict of figures."""
    import clip_tensor_adamw_gb300 as mica
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    W = mica.TensorList(st.w)
    G = mica.TensorList(st.g)
    M = mica.TensorList(st.m, W.counts)
    V = mica.TensorList(st.v, W.counts)
    norm = torch.empty(1, device="cuda")
    factor = torch.empty(1, device="cuda")
    kw = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay,
              zero_grad=zero_grad, factor=factor, coupled_l2=coupled_l2)
    stream = torch.cuda.current_stream()

    if opt == "adamw_groups":
        group, hps = decay_groups(wl)
        gi = mica.GroupIndex(group)
        gkw = dict(beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, zero_grad=zero_grad, factor=factor)

        def update(t):
            mica.mica_adamw_steps_grouped(W, G, M, V, gi, hps, step=t, **gkw)
    elif opt in ("sgd", "momentum"):
        B = M if opt == "momentum" else None
        mu = SGD_MOMENTUM if opt == "momentum" else 0.0

        def update(t):
            mica.mica_sgd_steps(W, G, B, lr=SGD_LR, momentum=mu, zero_grad=zero_grad, factor=factor)
    else:
        def update(t):
            mica.mica_adamw_steps(W, G, M, V, step=t, **kw)
    if opt == "accumulate":  # a second contribution to every gradient, laid out as g
        a_flat = torch.empty_like(st.g_flat)
        a_flat.normal_(0.0, wl.g_std, generator=torch.Generator(device="cuda").manual_seed(wl.seed + 1))
        es = st.g_flat.element_size()
        A = mica.TensorList([a_flat.narrow(0, (x.data_ptr() - st.g_flat.data_ptr()) // es, x.numel())
                             if x.numel() else a_flat[:0] for x in st.g])

    step_kw = dict(max_norm=wl.max_norm, inv_scale=wl.inv_scale, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                   weight_decay=wl.weight_decay, zero_grad=zero_grad, norm_out=norm, factor_out=factor,
                   coupled_l2=coupled_l2)

    def step(t, ev_mid=None):
        if ev_mid is None and opt == "adamw":  # the whole step through the one-step entry point
            mica.mica_clip_adamw_step(W, G, M, V, step=t, **step_kw)
            return
        if opt == "accumulate":
            mica.mica_accumulate_clip_grad_norms(G, A, wl.max_norm, wl.inv_scale, norm_out=norm, factor_out=factor)
        else:
            mica.mica_clip_grad_norms(G, wl.max_norm, wl.inv_scale, norm_out=norm, factor_out=factor)
        if ev_mid is not None:
            ev_mid.record(stream)
        update(t)

    for t in range(1, warmup + 1):
        step(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed region: K steps back to back, events only at its two ends
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = mica.mica_launch_count()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(steps):
        step(warmup + 1 + i)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    launches = mica.mica_launch_count() - launches0
    total_ms = start.elapsed_time(end)
    if dist is not None:
        dist.barrier()
        total_ms = slowest_rank_ms(total_ms, dist, "cuda")
    # each kernel's own duration, from events around each launch (a separate loop: events between the two
    # launches of a step keep them from overlapping)
    k2 = min(steps, 50) if per_kernel else 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(k2)]
    for i in range(k2):
        ev[i][0].record(stream)
        step(warmup + steps + 1 + i, ev[i][1])
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    adamw_ms = [e[1].elapsed_time(e[2]) for e in ev] or [float("nan")]
    clip_ms = [e[0].elapsed_time(e[1]) for e in ev] or [float("nan")]
    out = {"total_ms": total_ms, "ms_per_step": total_ms / steps, "steps": steps,
           "adamw_ms": statistics.mean(adamw_ms), "clip_ms": statistics.mean(clip_ms), "launches": launches,
           "t_wall": (t_wall0, t_wall1), "norm": float(norm.item())}
    mica.mica_sync()
    if opt == "accumulate":
        del A, a_flat
    del st, W, G, M, V
    mica.mica_release_cache()  # the list's tables go with its tensors
    torch.cuda.empty_cache()
    return out


def measure_scale(wl: workloads.Workload, steps: int, warmup: int) -> float:
    """ScaleTensors alone over the workload's gradient list: the mean device time of one call (ms), from events around
    `steps` back-to-back calls (factors 2 and 0.5 in turn, so the values stay as they were)."""
    import clip_tensor_adamw_gb300 as mica
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    G = mica.TensorList(st.g)
    for i in range(warmup):
        mica.mica_scale_tensors(G, 2.0 if i % 2 == 0 else 0.5)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(steps):
        mica.mica_scale_tensors(G, 2.0 if i % 2 == 0 else 0.5)
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    del st, G
    mica.mica_release_cache()
    torch.cuda.empty_cache()
    return ms


def measure_sharded(wl: workloads.Workload, steps: int, warmup: int, dist, world: int, rank: int):
    """The sharded step (the list split over the ranks, ZeRO-style): each rank's square sum of its own part
    (mica_grad_sumsq), an all-gather of one double per rank, the factor from the sums in rank order
    (mica_clip_factor_from_sumsq), and each rank's update of its own part. Times `steps` steps as measure() does."""
    import clip_tensor_adamw_gb300 as mica
    from clip_tensor_adamw_gb300.shard import piece_views, shard_pieces
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    pieces = shard_pieces(st.sizes, world, rank)
    counts = [b - a for _, a, b in pieces]
    W = mica.TensorList(piece_views(st.w, pieces))
    G = mica.TensorList(piece_views(st.g, pieces))
    M = mica.TensorList(piece_views(st.m, pieces, st.m_packed), counts)
    V = mica.TensorList(piece_views(st.v, pieces, st.packed), counts)
    mine = torch.zeros(1, dtype=torch.float64, device="cuda")
    parts = torch.zeros(world, dtype=torch.float64, device="cuda")
    norm = torch.empty(1, device="cuda")
    factor = torch.empty(1, device="cuda")
    kw = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay, factor=factor)
    stream = torch.cuda.current_stream()

    def step(t):
        mica.mica_grad_sumsq(G, wl.inv_scale, out=mine)
        if dist is not None:
            dist.all_gather_into_tensor(parts, mine)
        else:
            parts.copy_(mine)
        mica.mica_clip_factor_from_sumsq(parts, wl.max_norm, wl.inv_scale, norm_out=norm, factor_out=factor)
        mica.mica_adamw_steps(W, G, M, V, step=t, **kw)

    for t in range(1, warmup + 1):
        step(t)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = mica.mica_launch_count()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(steps):
        step(warmup + 1 + i)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    launches = mica.mica_launch_count() - launches0
    total_ms = start.elapsed_time(end)
    if dist is not None:
        dist.barrier()
        total_ms = slowest_rank_ms(total_ms, dist, "cuda")
    out = {"total_ms": total_ms, "ms_per_step": total_ms / steps, "steps": steps, "launches": launches,
           "t_wall": (t_wall0, t_wall1), "norm": float(norm.item()),
           "part_params": sum(counts), "pieces": len(pieces)}
    mica.mica_sync()
    del st, W, G, M, V
    mica.mica_release_cache()
    torch.cuda.empty_cache()
    return out


def measure_e2e(wl: workloads.Workload, steps: int, warmup: int):
    """The same step through the public API, fed from the host: every step copies its whole gradient from pinned host
    memory into one of two device gradient buffers (on a copy stream, so that step t+1's copy overlaps step t's
    kernels, as a training loop's input pipeline would) and reads the step's norm back into pinned host memory.
    Both copies of every step are inside the timed region. Returns (ms per step, H2D bytes, D2H bytes)."""
    import clip_tensor_adamw_gb300 as mica
    st = workloads.make_state(wl, "cuda")
    workloads.fill_grad(st, 1)
    g_host = torch.empty(st.g_flat.shape, dtype=st.g_flat.dtype, pin_memory=True)
    g_host.copy_(st.g_flat)
    g_flat = [st.g_flat, torch.empty_like(st.g_flat)]
    g_lists = [mica.TensorList(st.g)]
    views = [g_flat[1][(x.data_ptr() - st.g_flat.data_ptr()) // x.element_size():][:x.numel()] for x in st.g]
    g_lists.append(mica.TensorList(views))
    norm_host = torch.empty(2, dtype=torch.float32, pin_memory=True)
    W = mica.TensorList(st.w)
    M = mica.TensorList(st.m, W.counts)
    V = mica.TensorList(st.v, W.counts)
    norm = torch.empty(1, device="cuda")
    factor = torch.empty(1, device="cuda")
    kw = dict(max_norm=wl.max_norm, inv_scale=wl.inv_scale, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
              weight_decay=wl.weight_decay, norm_out=norm, factor_out=factor)
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    released = [torch.cuda.Event(), torch.cuda.Event()]
    for e in released:
        e.record(compute)

    def step(t):
        x = t % 2
        with torch.cuda.stream(copier):
            copier.wait_event(released[x])              # the buffer's previous step has read it
            g_flat[x].copy_(g_host, non_blocking=True)
            copied[x].record(copier)
        compute.wait_event(copied[x])
        mica.mica_clip_adamw_step(W, g_lists[x], M, V, step=t, **kw)
        released[x].record(compute)
        norm_host[x:x + 1].copy_(norm, non_blocking=True)

    for t in range(1, warmup + 1):
        step(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    copier.wait_event(e0)
    for i in range(steps):
        step(warmup + 1 + i)
    e1.record(compute)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = st.g_flat.numel() * st.g_flat.element_size()
    del st, g_flat, views, g_lists, W, M, V, g_host
    mica.mica_release_cache()
    torch.cuda.empty_cache()
    return ms, h2d, 4


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gpt2_small", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="mica", choices=["mica", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads, e2e and the CPU baseline")
    ap.add_argument("--shard", action="store_true",
                    help="split the list over the ranks (each steps its own part; one all-gather of the norm's "
                         "square sums a step) instead of stepping a replica on every rank")
    ap.add_argument("--step", default="clip_adamw", choices=["clip_adamw", "accumulate"],
                    help="the timed step: the norm then AdamW (default), or g += a with the norm fused into that "
                         "add, then AdamW (for profiling that kernel)")
    ap.add_argument("--subset-params", type=int, default=0,
                    help="keep only the workload's first tensors up to this many parameters (small profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = workloads.WORKLOADS[args.workload]
    if args.subset_params:
        shapes, tot = [], 0
        for s_, n in zip(wl.shapes, wl.sizes):
            if shapes and tot + n > args.subset_params:
                break
            shapes.append(s_)
            tot += n
        wl = dataclasses.replace(wl, name=f"{wl.name}[first {len(shapes)} tensors]", shapes=tuple(shapes))

    if args.impl == "reference":
        run_reference(args, wl)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    if world != args.gpus and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)

    import clip_tensor_adamw_gb300 as mica
    mica.lib()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if args.shard:
        main_fig = measure_sharded(wl, args.steps, args.warmup, dist, world, rank)
    else:
        main_fig = measure(wl, args.steps, args.warmup, zero_grad=False, dist=dist,
                           opt="accumulate" if args.step == "accumulate" else "adamw")
    if sampler:
        sampler.stop()
    clocks = sampler.summary(*main_fig["t_wall"]) if sampler else None
    if args.shard:
        if rank == 0:
            P = wl.params
            sec = main_fig["total_ms"] / 1e3
            gbs = P * step_bytes_per_param(wl) * args.steps / sec / 1e9
            print(json.dumps({
                "metric": METRIC, "value": P * args.steps / sec, "unit": "params/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_fig["ms_per_step"],
                "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": {**run_config(wl, world), "parallelism": f"sharded x{world} (one all-gather a step)"},
                "hbm_gbs": gbs, "pct_of_8tbs": 100 * gbs / NOMINAL_HBM_GBS, "clocks": clocks,
                "gpu_launches": main_fig["launches"], "norm": main_fig["norm"],
                "rank0_part_params": main_fig["part_params"]}), flush=True)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return

    P = wl.params
    sec = main_fig["total_ms"] / 1e3
    value = job_value(world, P, args.steps, main_fig["total_ms"])
    step_bpp = step_bytes_per_param(wl, opt="accumulate" if args.step == "accumulate" else "adamw")
    step_gbs = P * step_bpp * args.steps / sec / 1e9
    a_bpp = adamw_bytes_per_param(wl)
    a_gbs = P * a_bpp / (main_fig["adamw_ms"] / 1e3) / 1e9
    peak, peak_src = hbm_peak()

    extras = {}
    e2e = None
    cpu = None
    if not args.no_extras and rank == 0:
        zg = measure(wl, extra_steps(main_fig["ms_per_step"]), args.warmup, zero_grad=True)
        extras["zero_grad"] = {"ms_per_step": zg["ms_per_step"], "steps": zg["steps"],
                               "hbm_gbs_model": P * step_bytes_per_param(wl) / (zg["ms_per_step"] / 1e3) / 1e9,
                               "hbm_gbs_actual": P * step_bytes_per_param(wl, True) / (zg["ms_per_step"] / 1e3) / 1e9,
                               "bytes_per_param_actual": step_bytes_per_param(wl, True)}
        small = workloads.WORKLOADS["gpt2_small"]
        others = [(n, workloads.WORKLOADS[n], False, "adamw", None)
                  for n in ("gpt2_small_bf16", "gpt2_xl", "fp16_scaled", "tiny")]
        others += [("fp16_scaled_cooperative", workloads.WORKLOADS["fp16_scaled"], False, "adamw", "1"),
                   ("gpt2_small_bf16_m", dataclasses.replace(small, name="gpt2_small_bf16_m", moments="bf16x2_m"),
                    False, "adamw", None),
                   ("gpt2_small_adam_l2", small, True, "adamw", None),
                   ("gpt2_small_param_groups", small, False, "adamw_groups", None),
                   ("gpt2_small_accumulate", small, False, "accumulate", None),
                   ("gpt2_small_sgd", small, False, "sgd", None),
                   ("gpt2_small_sgd_momentum", small, False, "momentum", None)]
        for other, owl, coupled, opt, fused in others:
            if other == wl.name:
                continue
            if fused is not None:
                os.environ["MICA_FUSED"] = fused
            est = measure(owl, 10, args.warmup, zero_grad=False, coupled_l2=coupled, opt=opt, per_kernel=False)
            f = measure(owl, extra_steps(est["ms_per_step"]), args.warmup, zero_grad=False, coupled_l2=coupled,
                           opt=opt)
            os.environ.pop("MICA_FUSED", None)
            torch.cuda.empty_cache()
            bpp = step_bytes_per_param(owl, opt=opt)
            ubpp = adamw_bytes_per_param(owl, opt=opt)
            extras[other] = {"params": owl.params, "steps": f["steps"], "ms_per_step": f["ms_per_step"],
                             "params_per_s": owl.params / (f["ms_per_step"] / 1e3),
                             "hbm_gbs": owl.params * bpp / (f["ms_per_step"] / 1e3) / 1e9,
                             "pct_of_8tbs": 100 * owl.params * bpp / (f["ms_per_step"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                             "update_ms": f["adamw_ms"], "clip_ms": f["clip_ms"], "bytes_per_param": bpp,
                             "update_gbs": owl.params * ubpp / (f["adamw_ms"] / 1e3) / 1e9,
                             "roofline": {"bound": "hbm", "kernel": "sgd_kernel" if opt in ("sgd", "momentum")
                                          else "adamw_kernel", "achieved": owl.params * ubpp / f["adamw_ms"] / 1e6,
                                          "peak": peak, "unit": "GB/s",
                                          "frac": owl.params * ubpp / f["adamw_ms"] / 1e6 / peak,
                                          "peak_source": peak_src, "bytes_per_param": ubpp,
                                          "launch_ms": f["adamw_ms"]}}
            if fused is not None:
                extras[other]["path"] = "one cooperative launch (MICA_FUSED=1)"
            if opt == "accumulate":  # the add + norm kernel: reads g and a, writes g
                abpp = 3 * (2.0 if owl.grad_dtype == "f16" else 4.0)
                extras[other]["path"] = "g += a with the norm fused into the add, then AdamWSteps"
                extras[other]["accumulate_kernel"] = {
                    "kernel": "accumulate_norm_kernel", "launch_ms": f["clip_ms"], "bytes_per_param": abpp,
                    "achieved": owl.params * abpp / f["clip_ms"] / 1e6, "peak": peak, "unit": "GB/s",
                    "frac": owl.params * abpp / f["clip_ms"] / 1e6 / peak, "peak_source": peak_src}
            if other == "gpt2_xl":
                ms, h2d, d2h = measure_e2e(owl, 10, args.warmup)
                extras[other]["e2e"] = {"value": owl.params / (ms / 1e3), "unit": "params/s", "ms_per_step": ms,
                                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
                params, ntens, times = time_oracle(owl, target_params=owl.params // 8, min_seconds=5.0, max_steps=5)
                extras[other]["cpu_baseline"] = {
                    "value": params * len(times) / sum(times), "unit": "params/s", "cores": 1, "kind": "oracle",
                    "host": host_cpu(),
                    "sample": f"{len(times)} steps of the first {ntens} of {len(owl.sizes)} tensors ({params:,} of "
                              f"{owl.params:,} params) of {owl.name}, single-threaded C oracle"}
                torch.cuda.empty_cache()
        for sname, swl in (("scale_tensors_fp16_scaled", workloads.WORKLOADS["fp16_scaled"]),
                           ("scale_tensors_gpt2_small", small)):
            sms_ = measure_scale(swl, extra_steps(0.1), args.warmup)
            sbpp = 2 * (2.0 if swl.grad_dtype == "f16" else 4.0)  # each cell read and written
            extras[sname] = {"params": swl.params, "ms_per_call": sms_, "bytes_per_param": sbpp,
                             "roofline": {"bound": "hbm", "kernel": "scale_kernel",
                                          "achieved": swl.params * sbpp / sms_ / 1e6, "peak": peak, "unit": "GB/s",
                                          "frac": swl.params * sbpp / sms_ / 1e6 / peak, "peak_source": peak_src,
                                          "bytes_per_param": sbpp, "launch_ms": sms_}}
        ms, h2d, d2h = measure_e2e(wl, extra_steps(main_fig["ms_per_step"]), args.warmup)
        e2e = {"value": P / (ms / 1e3), "unit": "params/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}
        params, ntens, times = time_oracle(wl, target_params=wl.params, min_seconds=10.0, max_steps=20)
        cpu = {"value": params * len(times) / sum(times), "unit": "params/s", "cores": 1, "kind": "oracle",
               "host": host_cpu(),
               "sample": f"{len(times)} full steps of the first {ntens} of {len(wl.sizes)} tensors "
                         f"({params:,} params) of {wl.name}, single-threaded C oracle"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": main_fig["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(run_config(wl, world), **({"step": "g += a with the norm fused, then AdamW",
                                                       "bytes_per_param": step_bpp}
                                                      if args.step == "accumulate" else {})),
            "hbm_gbs": step_gbs, "pct_of_8tbs": 100 * step_gbs / NOMINAL_HBM_GBS,
            "pct_of_measured_copy": 100 * step_gbs / peak if peak_src == "measured" else None,
            "roofline": {"bound": "hbm", "kernel": "adamw_kernel", "achieved": a_gbs, "peak": peak, "unit": "GB/s",
                         "frac": a_gbs / peak, "peak_source": peak_src, "traffic": profiled_traffic(),
                         "bytes_per_param": a_bpp, "launch_ms": main_fig["adamw_ms"]},
            "clip_ms": main_fig["clip_ms"], "norm": main_fig["norm"],
            "clocks": clocks, "gpu_launches": main_fig["launches"],
            "e2e": e2e, "cpu_baseline": cpu, "also": extras,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
