"""Benchmark of one Muon optimizer step on synthetic data (prints ONE JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--ns-dtype bf16|fp32|split]
    python bench.py --impl reference ...   # the fp64 CPU oracle on this host's cores

A step is the whole hot path over one flat buffer: momentum + orthogonalization input +
gather + Frobenius norms, 5 Newton-Schulz iterations (15 grouped tcgen05 GEMM launches),
then decay + scaled update + scatter.  The default workload is the Llama-3-8B matrix set
(32 layers x {q, o, k, v, gate, up, down}, 224 matrices, 6.98e9 fp32 elements per
buffer), whose buffers are far larger than L2, so no flush is needed between steps.

Under torchrun (N > 1) every rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon step time (ms) and Newton\u2013Schulz TFLOP/s + % bf16 peak at 1 GB300"
DEFAULT_WORKLOAD = "llama3_8b_x32"


def ns_flops(shapes, is_matrix, ns_steps):
    """(symmetric, dense) Newton-Schulz flop counts of one step.

    Per iteration and matrix (m = min, n = max of the shape), in multiply-adds: the Gram
    X X^T on its upper half m^2 n / 2, A A on its upper half m^3 / 2, B X m^2 n; 2 flops per
    multiply-add gives 3 m^2 n + m^3 (symmetric) against 4 m^2 n + 2 m^3 (dense).
    """
    sym = dense = 0.0
    for (r, c), f in zip(shapes, is_matrix):
        if not f:
            continue
        m, n = min(r, c), max(r, c)
        sym += ns_steps * (3.0 * m * m * n + m ** 3)
        dense += ns_steps * (4.0 * m * m * n + 2.0 * m ** 3)
    return sym, dense


def elementwise_bytes(n_matrix_elems, ns_dtype):
    """Algorithmic HBM bytes of the two streaming passes per step.

    Stage 1 reads G and M and writes M (12 B) and X (2 B bf16 / 4 B fp32 / 6 B as three
    bf16 parts); stage 3 reads W and O (2 / 4 / 6 B) and writes W (8 B): 24 B per element
    on the bf16 path."""
    x = {"bf16": 2, "fp32": 4, "split": 6}[ns_dtype]
    return n_matrix_elems * (12 + x), n_matrix_elems * (8 + x)


# DRAM bytes per Newton-Schulz launch (mean over the 15 launches of one step: Gram, Poly,
# Update x 5, the last Update also applying W), measured with ncu on two Llama-3-8B layers
# with the same kernel shape and scaled by 16 to the 32-layer set.  Valid only for the
# kernel shape and the sources it was taken with.
NS_TRAFFIC = {
    # single-CTA tiles with the fused tail, as the 32-layer set runs (MUON_TC_KERNEL=1
    # MUON_FUSED_TAIL=1 on two layers): 19.48 GB read + 8.90 GB written over 15 launches
    "llama3_8b_x32": {"bytes_per_launch": 16 * (19478732800 + 8900310528) / 15,
                      "tile_shape": 1,
                      "sources_sha256": "7e1b55959783a9afe198de808c4756547116d015e608b3e7e6ec3a71accbdcf3"},
}
NS_SOURCES = ("gemm_ns.cu", "device_common.cuh", "layout.cpp")


def _ns_sources_sha256():
    """Digest of the kernel sources' code: comments and whitespace are dropped, so that a
    change of wording alone keeps the measured traffic."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in NS_SOURCES:
        with open(os.path.join(ROOT, "muon_optimizer_step_gb300", "csrc", f)) as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()


def ns_traffic(workload, ns_dtype, kernel):
    """Measured DRAM bytes per Newton-Schulz launch, or None if not measured for this
    workload and kernel shape, or if the kernel sources changed since the counters were
    taken."""
    rec = NS_TRAFFIC.get(workload)
    if rec is None or ns_dtype != "bf16" or kernel is None:
        return None
    if kernel["tile_shape"] != rec["tile_shape"]:
        return None
    try:
        if _ns_sources_sha256() != rec["sources_sha256"]:
            return None
    except OSError:
        return None
    return rec["bytes_per_launch"]


NS_KERNEL_NAMES = {
    1: "ns_tc_single_kernel (tcgen05 cta_group::1, 128x256 tiles)",
    2: "ns_tc_pair_kernel (tcgen05 cta_group::2, 256x256 tiles)",
    3: "ns_tc_pairwide_kernel (tcgen05 cta_group::2, 256x512 tiles)",
}


def ns_kernel_label(kernel, ns_steps, ns_dtype="bf16", fused=False):
    if kernel is None:
        return "ns_phase_f32_kernel (fp32 CUDA cores, 3 launches per iteration)"
    launches = 1 if kernel["persistent"] else 3 * ns_steps
    name = NS_KERNEL_NAMES[kernel["tile_shape"]] if ns_dtype == "bf16" else \
        "ns_tc_split_kernel (tcgen05 cta_group::2, fp32 as 3 bf16 parts, 6 products, " \
        "256x256 tiles)"
    return "%s, %d units, %d launch(es) per step; %s" % (
        name, kernel["units"], launches,
        "the last Update also applies W" if fused else "a separate apply pass follows (timed apart)")


# Process-group timeout of the multi-rank bench: far above any step, far below forever.
PG_TIMEOUT_S = 600


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "sm_mhz_under_load": (p.get("clocks_under_load") or {}).get("sm_mhz_median"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_mhz_under_load": None, "source": "fallback"}


def per_mhz(tflops, sm_mhz, peaks):
    """TFLOP/s per MHz of SM clock, next to the cuBLAS sustained figure per MHz of the clock
    it ran at, so that a clock advantage is not read as kernel efficiency."""
    ref_mhz = peaks.get("sm_mhz_under_load")
    out = {"ns_tflops_per_mhz": tflops / sm_mhz if sm_mhz else None,
           "cublas_sustained_tflops_per_mhz":
               peaks["bf16_tflops_sustained"] / ref_mhz if ref_mhz else None,
           "ns_sm_mhz": sm_mhz, "cublas_sm_mhz": ref_mhz}
    if out["ns_tflops_per_mhz"] and out["cublas_sustained_tflops_per_mhz"]:
        out["ratio"] = out["ns_tflops_per_mhz"] / out["cublas_sustained_tflops_per_mhz"]
    return out


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_matrix_step_seconds(r, c, seed, ns_steps=5):
    """Seconds the fp64 oracle takes for one full step of one r x c matrix."""
    import numpy as np
    from oracle import muon_ref as ref
    rng = np.random.default_rng(seed)
    W = rng.normal(0.0, 0.02, r * c)
    G = rng.normal(0.0, 1e-3, r * c)
    M = np.zeros(r * c)
    lay = ref.flat_layout([(r, c)], 1)
    t0 = time.perf_counter()
    ref.muon_step(W, G, M, lay, 0.02, 0.01, 0.95, True, ns_steps)
    return time.perf_counter() - t0


def _shape_classes(wl):
    """Distinct matrix costs: a matrix and its transpose share one class."""
    classes = {}
    for (r, c), f in zip(wl.shapes, wl.is_matrix):
        if f:
            key = (max(r, c), min(r, c))
            classes[key] = classes.get(key, 0) + 1
    return classes


def bench_config(wl, ns_dtype):
    """The workload description both arms print (identical for the same arguments)."""
    n = wl.numel
    l2 = ("inputs larger than L2 (%.1f GB per fp32 buffer); no flush" % (4 * n / 1e9)
          if 4 * n > 129e6 else
          "inputs smaller than L2 (%.1f MB per fp32 buffer); no flush" % (4 * n / 1e6))
    return {"workload": wl.name, "matrices": wl.n_matrices, "elements": n,
            "n_shards": wl.n_shards, "ns_steps": wl.ns_steps, "ns_dtype": ns_dtype, "l2": l2}


def _cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def _estimate(classes, times):
    """Whole-step estimate: every shape class's mean one-matrix time x its matrix count."""
    return sum(count * statistics.mean(times[key]) for key, count in classes)


def _method(wl, ns_steps):
    return (f"fp64 numpy oracle: one full step (momentum, {ns_steps} Newton-Schulz iterations, "
            f"apply) of one matrix per distinct shape class (a matrix and its transpose share "
            f"a class), each class's mean time x its matrix count, summed over the "
            f"{len(_shape_classes(wl))} classes of the {wl.n_matrices}-matrix workload")


def cpu_baseline(wl, ns_steps):
    """The oracle on one matrix of each distinct shape, extrapolated to the whole step by
    the shape counts (the same method as the reference arm)."""
    classes = sorted(_shape_classes(wl).items(), key=lambda kv: kv[0][0] * kv[0][1])
    times = {}
    spent = 0.0
    for (n, m), _ in classes:
        t = _oracle_matrix_step_seconds(n, m, seed=n + m, ns_steps=ns_steps)
        times[(n, m)] = [t]
        spent += t
    return {"value": _estimate(classes, times) * 1e3, "unit": "ms", "cores": _cores(),
            "kind": "oracle",
            "sample": _method(wl, ns_steps) + f"; one pass over the classes, {spent:.1f} s of CPU work",
            "sample_seconds": spent}


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on this host's cores.

    Each timed step is a bounded sample: one matrix step of one shape class, the classes
    taken in turn (all classes in every step when there are fewer steps than classes).
    The line reports the whole-step estimate built from those samples, the same method as
    the cpu_baseline leg of the GPU arm."""
    from muon_optimizer_step_gb300 import inputs
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = inputs.WORKLOADS[args.workload]
    ns_steps = wl.ns_steps
    classes = sorted(_shape_classes(wl).items(), key=lambda kv: kv[0][0] * kv[0][1])
    small = classes[0][0]
    for _ in range(args.warmup):  # warms the BLAS threads on the cheapest class
        _oracle_matrix_step_seconds(small[0], small[1], 7, ns_steps)
    times = {key: [] for key, _ in classes}
    per_step = []
    t_all = time.perf_counter()
    for k in range(args.steps):
        todo = [classes[k % len(classes)][0]] if args.steps >= len(classes) else \
            [key for key, _ in classes]
        t0 = time.perf_counter()
        for (n, m) in todo:
            times[(n, m)].append(_oracle_matrix_step_seconds(n, m, 7 + k, ns_steps))
        per_step.append(time.perf_counter() - t0)
    wall = time.perf_counter() - t_all
    ms = _estimate(classes, times) * 1e3
    cores = _cores()
    sample = (_method(wl, ns_steps) + f"; {args.steps} timed steps, each one bounded sample "
              f"(one class in turn), {wall:.1f} s of CPU work")
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": "ms",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(wl, args.ns_dtype),
            "sample_seconds_per_step": per_step,
            "cpu_baseline": {"value": ms, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": ms, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def _mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def host_memory_allows(need_bytes, world, dist, device, available=None):
    """Whether every rank may pin `need_bytes` of host memory.  The ranks share one host:
    each asks for room for all of them (three times the total, for headroom), and all
    skip together when any rank sees too little."""
    avail = _mem_available_bytes() if available is None else available
    short = 0.0 if avail > 3 * need_bytes * world else 1.0
    return reduce_max_over_ranks([short], dist, device)[0] == 0.0


def _pin_to_gpu_numa_node(dev):
    """Run this thread on the CPUs next to the GPU, so pinned pages land on its node."""
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        if cpus:
            os.sched_setaffinity(0, cpus)
    except (OSError, AttributeError, ValueError):
        pass


def reduce_max_over_ranks(values, dist, device):
    """Element-wise max of a list of floats over all ranks (the timing rule: the slowest
    rank sets the step time); identity without a process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def run_ours(args):
    import torch
    from muon_optimizer_step_gb300 import capi, inputs

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        # A rank that dies must not hold the others forever: their next collective
        # fails after this timeout (tested on gloo ranks in tests/test_owners_and_ranks.py).
        dist.init_process_group("nccl", device_id=torch.device("cuda", local),
                                timeout=datetime.timedelta(seconds=PG_TIMEOUT_S))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    wl = inputs.WORKLOADS[args.workload]
    ns_dtype = {"bf16": capi.MUON_NS_BF16, "fp32": capi.MUON_NS_FP32,
                "split": capi.MUON_NS_SPLIT_FP32}[args.ns_dtype]
    ns_steps = wl.ns_steps
    lay = capi.muon_layout_create(wl.shapes, wl.n_shards, ns_dtype, wl.is_matrix)
    ns_kernel = capi.muon_layout_ns_kernel(lay) if ns_dtype != capi.MUON_NS_FP32 else None
    S, L, N = wl.n_shards, lay.shard_len, lay.numel
    # One allocation per buffer; shard s is a view of [s*L, (s+1)*L), the first N elements
    # are the unsharded flat buffer.
    Wb = torch.zeros(S * L, dtype=torch.float32, device=dev)
    Gb = torch.zeros(S * L, dtype=torch.float32, device=dev)
    Mb = torch.zeros(S * L, dtype=torch.float32, device=dev)
    inputs.device_fill_weights(wl, Wb[:N])
    inputs.device_fill_grads(wl, Gb[:N], 0)
    W = [Wb[s * L:(s + 1) * L] for s in range(S)]
    G = [Gb[s * L:(s + 1) * L] for s in range(S)]
    M = [Mb[s * L:(s + 1) * L] for s in range(S)]
    ws = capi.workspace_tensor(lay, dev)
    torch.cuda.synchronize()

    # One timed step = the launches muon_step makes, through the public calls that split
    # them into stages, with events between the stages: stage 1 (momentum and the
    # Newton-Schulz input), then the Newton-Schulz launches, then the apply pass - or,
    # where the library applies W inside the last Update, stages 2 and 3 as one call.
    n_mat_elems = sum(r * c for (r, c), f in zip(wl.shapes, wl.is_matrix) if f)
    fused = (ns_steps >= 1 and args.ns_dtype != "fp32" and n_mat_elems > 0
             and capi.muon_layout_fused_apply(lay))

    def step_stages(evs=None):
        if evs is not None:
            evs[0].record()
        capi.muon_compute_momentum_inputs(G, M, lay, ws, wl.mu, wl.nesterov)
        if evs is not None:
            evs[1].record()
        if fused:
            capi.muon_orthogonalize_apply(W, lay, ws, wl.lr, wl.wd, ns_steps)
            if evs is not None:
                evs[2].record()
                evs[3].record()
        else:
            capi.muon_orthogonalize_updates(lay, ws, ns_steps)
            if evs is not None:
                evs[2].record()
            capi.muon_apply_local_updates(W, lay, ws, wl.lr, wl.wd, ns_steps)
            if evs is not None:
                evs[3].record()

    for _ in range(args.warmup):
        step_stages()
    capi.muon_check()

    def barrier():
        if dist is not None:
            dist.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    t_start.record()
    for k in range(args.steps):
        step_stages(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    barrier()
    capi.muon_check()
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = [0.0, 0.0, 0.0]
    for e in evs:
        for j in range(3):
            stage_ms[j] += e[j].elapsed_time(e[j + 1])
    stage_ms = [x / args.steps for x in stage_ms]
    red = reduce_max_over_ranks([total_ms] + stage_ms, dist, dev)
    total_ms, stage_ms = red[0], red[1:]
    ms = total_ms / args.steps

    # ------------------------------------------------------------ end to end (host buffers)
    # Every step takes its gradient from pinned host memory and returns its updated
    # weights to pinned host memory, through the same public calls the timed step makes
    # (stage 1, then the orthogonalization whose last Update applies W).  The copies of
    # neighbouring steps are pipelined on two copy streams: step t+1's gradient goes up
    # while step t runs; step t's weights are snapshot on the device (a device copy right
    # after the step, so that step t+1 may update W while they travel) and go down while
    # step t+1 runs.
    e2e = None
    if not args.no_e2e:
        need = 2 * 4 * N
        barrier()
        if host_memory_allows(need, world, dist, dev):
            saved_affinity = os.sched_getaffinity(0)
            _pin_to_gpu_numa_node(dev)
            G_h = torch.empty(N, dtype=torch.float32, pin_memory=True)
            W_h = torch.empty(N, dtype=torch.float32, pin_memory=True)
            G_h.copy_(Gb[:N])
            os.sched_setaffinity(0, saved_affinity)
            G2b = torch.empty_like(Gb)
            W_snap = torch.empty(N, dtype=torch.float32, device=dev)
            gbufs = [Gb, G2b]
            h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
            comp = torch.cuda.current_stream()
            n_e2e = max(2, args.steps)
            ev = lambda: torch.cuda.Event()  # noqa: E731
            ev_in = [ev(), ev()]
            ev_k1 = [ev(), ev()]
            ev_snap = [ev() for _ in range(n_e2e)]
            ev_out = [ev() for _ in range(n_e2e)]
            torch.cuda.synchronize()
            barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(comp)
            h2d.wait_stream(comp)
            with torch.cuda.stream(h2d):
                gbufs[0][:N].copy_(G_h, non_blocking=True)
                ev_in[0].record(h2d)
            for t in range(n_e2e):
                cur = gbufs[t % 2]
                shards = [cur[s * L:(s + 1) * L] for s in range(S)]
                comp.wait_event(ev_in[t % 2])
                capi.muon_compute_momentum_inputs(shards, M, lay, ws, wl.mu, wl.nesterov)
                ev_k1[t % 2].record(comp)
                if t + 1 < n_e2e:
                    with torch.cuda.stream(h2d):
                        if t >= 1:
                            h2d.wait_event(ev_k1[(t + 1) % 2])
                        gbufs[(t + 1) % 2][:N].copy_(G_h, non_blocking=True)
                        ev_in[(t + 1) % 2].record(h2d)
                capi.muon_orthogonalize_apply(W, lay, ws, wl.lr, wl.wd, ns_steps)
                if t >= 1:
                    comp.wait_event(ev_out[t - 1])  # the snapshot buffer is free again
                W_snap.copy_(Wb[:N])
                ev_snap[t].record(comp)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(ev_snap[t])
                    W_h.copy_(W_snap, non_blocking=True)
                    ev_out[t].record(d2h)
            comp.wait_event(ev_out[n_e2e - 1])
            b.record(comp)
            torch.cuda.synchronize()
            e2e_ms = a.elapsed_time(b) / n_e2e
            e2e_ms = reduce_max_over_ranks([e2e_ms], dist, dev)[0]
            e2e = {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": 4 * N,
                   "d2h_bytes_per_step": 4 * N, "steps": n_e2e,
                   "note": "per step: gradient H2D from pinned host memory, "
                           "muon_compute_momentum_inputs + muon_orthogonalize_apply (the "
                           "calls muon_step makes), a device snapshot of W, W D2H to pinned "
                           "host memory; copies of neighbouring steps overlap compute on two "
                           "copy streams"}
            del G_h, W_h, G2b, W_snap
        else:
            e2e = {"value": None, "unit": "ms", "h2d_bytes_per_step": 4 * N,
                   "d2h_bytes_per_step": 4 * N,
                   "note": "not measured: not enough host memory to pin %.1f GB per rank "
                           "for %d rank(s)" % (need / 1e9, world)}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    sym, dense = ns_flops(wl.shapes, wl.is_matrix, ns_steps)
    b1, b3 = elementwise_bytes(n_mat_elems, args.ns_dtype)
    ns_ms = stage_ms[1]
    ns_tflops = sym / (ns_ms * 1e-3) / 1e12
    ew_ms = stage_ms[0]
    ew_gbs = b1 / (ew_ms * 1e-3) / 1e9
    if args.ns_dtype == "bf16":
        peak_tc = peaks["bf16_tflops_sustained"]
        peak_note = "%s bf16 sustained (cuBLAS loop under the power cap)" % peaks["source"]
    elif args.ns_dtype == "split":
        # six bf16 MMAs per useful product
        peak_tc = peaks["bf16_tflops_sustained"] / 6.0
        peak_note = ("%s bf16 sustained / 6 (six bf16 products per useful one)"
                     % peaks["source"])
    else:
        # fp32 FMA issue rate: 128 FP32 lanes per SM x 2 flops x SMs x max SM clock.
        props = torch.cuda.get_device_properties(dev)
        peak_tc = props.multi_processor_count * 128 * 2 * 2070e6 / 1e12
        peak_note = "derived fp32 CUDA-core peak: %d SMs x 128 lanes x 2 flops x 2070 MHz" % (
            props.multi_processor_count)
    ns_launches = (1 if ns_kernel is not None and ns_kernel["persistent"] else 3 * ns_steps) \
        if ns_steps >= 1 else 0
    # stage 1 (momentum + norm finalize), the Newton-Schulz launches, and the apply pass
    # unless the last Update applies W
    launches_per_step = (2 + ns_launches + (0 if fused else 1)) if n_mat_elems else 0
    line = {
        "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": args.ns_dtype,
        "dtype_detail": "fp32 weights, momentum and update arithmetic; Newton-Schulz on "
                        + {"bf16": "bf16 tensor-core operands with fp32 accumulation",
                           "fp32": "fp32 CUDA cores",
                           "split": "tensor cores, fp32 operands split into three bf16 "
                                    "parts, six bf16 products each, fp32 accumulation"}[args.ns_dtype],
        "data": "synthetic",
        "config": bench_config(wl, args.ns_dtype),
        "ns_ms": ns_ms, "ns_tflops": ns_tflops, "ns_tflops_dense_equiv": dense / (ns_ms * 1e-3) / 1e12,
        "ns_flops_sym": sym,
        # whole job: every rank steps its own replica in the (max over ranks) step time
        "matrices_per_s": world * wl.n_matrices / (ms * 1e-3),
        "stage_ms": ({"momentum_inputs": stage_ms[0], "orthogonalize_apply": stage_ms[1]}
                     if fused else
                     {"momentum_inputs": stage_ms[0], "newton_schulz": stage_ms[1],
                      "apply": stage_ms[2]}),
        "fused_apply": bool(fused),
        "roofline": {"bound": "alu" if args.ns_dtype == "fp32" else "tensor",
                     "kernel": ns_kernel_label(ns_kernel, ns_steps, args.ns_dtype, fused),
                     "achieved": ns_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": ns_tflops / peak_tc,
                     "frac_of_burst": (ns_tflops / peaks["bf16_tflops"]
                                       if args.ns_dtype == "bf16" else None),
                     "peak_burst": peaks["bf16_tflops"] if args.ns_dtype == "bf16" else None,
                     "per_mhz": (per_mhz(ns_tflops, (clocks or {}).get("sm_mhz"), peaks)
                                 if args.ns_dtype == "bf16" else None),
                     "traffic": ns_traffic(wl.name, args.ns_dtype, ns_kernel),
                     "traffic_unit": "DRAM bytes per launch (ncu, mean over phases)",
                     "peak_note": peak_note},
        "roofline_elementwise": {"bound": "hbm", "kernel": "momentum_input_kernel",
                                 "achieved": ew_gbs, "peak": peaks["hbm_gbs"],
                                 "unit": "GB/s", "frac": ew_gbs / peaks["hbm_gbs"],
                                 "bytes_per_step": b1},
        "roofline_apply": (None if fused else
                           {"bound": "hbm", "kernel": "apply_kernel",
                            "achieved": b3 / (stage_ms[2] * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                            "unit": "GB/s",
                            "frac": b3 / (stage_ms[2] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                            "bytes_per_step": b3}),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, ns_steps)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--ns-dtype", choices=["bf16", "fp32", "split"], default="bf16")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
