#!/usr/bin/env python
"""Benchmark of the GB300 MoE route-sort path (one JSON line on stdout).

Headline workload: Kimi-K3-shaped TP8 decode, T=1 token, E=896 experts, n_group=8,
topk_group=4, top-16, block_m=32 (``decode_T1_E896_G8``); value = device microseconds per
route-sort call.  The large-T workloads (T=512/E=896, T=8192/E=896 skewed,
T=16384/E=4096) are measured in the same run and reported under ``configs`` as routed
tokens/s and fraction of the HBM roofline.

Timing: a step is one CUDA graph of C calls, each the whole path (route step + both sort
phases) on its own input set and output set; the sets rotate so that their total is larger
than twice the L2, and L2 is flushed (a 256 MiB write) before every timed step.  Each step
is bracketed by CUDA events on the launching stream; warm-up steps are not timed; a
workload's figure is the median over its timed steps.  Under torchrun each rank times its own
replica (the path does not shard: replicas only), the step times are reduced with MAX over
ranks, ``value`` is the per-call latency of the slowest rank (never divided by the rank count)
and ``job_calls_per_s`` the whole job's call rate.  For the one-token headline,
``single_call`` also times one call alone (a graph of one call, L2 flushed) beside the same
measurement of a T = 0 call, the launch floor.

``--impl reference`` times the CPU oracle (single thread, the slow plain definition) on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_expert_routing_sort_gb300 import datagen  # noqa: E402

HEADLINE = "decode_T1_E896_G8"
SECONDARY = ["prefill_T512_E896", "skewed_T8192_E896", "wide_T16384_E4096"]
SWEEP_TOKENS = [2, 8, 64, 152, 192, 384, 768, 1024, 1536, 2048, 3072, 4096]
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024
METRIC = "route-sort µs/call at T=1 E=896; routed tokens/s and % HBM roofline at T≥512"
CSRC = os.path.join(ROOT, "moe_expert_routing_sort_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE, choices=list(datagen.WORKLOADS))
    p.add_argument("--no-secondary", action="store_true",
                   help="skip the large-T workloads reported under 'configs'")
    p.add_argument("--cpu-budget", type=float, default=10.0,
                   help="seconds of oracle work for the CPU baseline of the headline workload")
    return p.parse_args()


# ---------------------------------------------------------------------- helpers
def algorithmic_bytes(w, npp: int) -> int:
    """Logits + bias read, top-k ids/weights, sorted ids/weights, block owners, npp written."""
    return (2 * w.T * w.E + 4 * w.E + 8 * w.T * w.topk + 8 * npp + 4 * (npp // w.block_m) + 4)


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the CUDA sources, in name order: names the kernels a
    DRAM-traffic capture was taken on."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def captured_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the workload's dominant kernel from the ncu
    capture recorded in profiles/dram_traffic.txt, or None when no capture of the current
    kernel sources exists (a table row: | workload | kernel | bytes | source hash | ...)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = kernel_source_hash()
    with open(TRAFFIC_FILE) as f:
        for line in f:
            cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == workload and cells[3] == want:
                try:
                    return int(float(cells[2]))
                except ValueError:
                    return None
    return None


def cpu_info():
    """Host cores and CPU model, for the CPU baseline record."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in text.splitlines():
                if line.lower().startswith(key.lower()):
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                break
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "model": model or platform.machine()}


class OneCore:
    """Pin this process to one core while timing the single-threaded oracle."""

    def __enter__(self):
        self.saved = None
        if hasattr(os, "sched_getaffinity"):
            self.saved = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {min(self.saved)})
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)
        return False


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init(n_gpus: int):
    """Join the launcher's process group (NCCL with GPUs, gloo on a host without any)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return rank, world, local


def dist_max(value: float, world: int) -> float:
    """MAX of a per-rank value over all ranks (the slowest rank's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------- GPU timing
class Replica:
    """Rotating input/output sets of one workload on the current device."""

    def __init__(self, w, n_sets: int):
        import torch

        import moe_expert_routing_sort_gb300 as mrs

        self.w = w
        self.sets = []
        for i in range(n_sets):
            inp = datagen.make_inputs(dataclasses.replace(w, seed=w.seed + i))
            logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).cuda()
            bias = torch.from_numpy(inp.bias).cuda()
            out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device="cuda")
            self.sets.append((logits, bias, out))
        self.mrs = mrs

    def call(self, i: int, stream=None):
        logits, bias, out = self.sets[i]
        w = self.w
        self.mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                            w.block_m, out=out, stream=stream)

    def npp(self) -> list:
        return [int(o.num_tokens_post_pad.item()) for _, _, o in self.sets]


def launches_per_call(w) -> int:
    """Kernels one route-sort call launches: one for T <= 4 (the one-token or single-CTA
    kernel), two from 5 to 2048 tokens (the zeroing kernel and a cooperative grid), three
    above (route, slices, scatter)."""
    if w.T <= 4:
        return 1
    return 2 if w.T <= 2048 else 3


def time_graph_steps(rep: Replica, steps: int, warmup: int, world: int, clocks=None):
    """Time `steps` graph replays (all sets once per step), L2 flushed before each step."""
    import torch

    s = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(s):
        for i in range(len(rep.sets)):
            rep.call(i)  # first calls outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(len(rep.sets)):
            rep.call(i)
    with torch.cuda.stream(s):
        for _ in range(warmup):
            flush.fill_(1)
            g.replay()
    torch.cuda.synchronize()
    if clocks is not None:
        # soak: keep the same work running ~1 s so the sampled clocks reflect it
        t_end = time.time() + 1.0
        while time.time() < t_end:
            with torch.cuda.stream(s):
                for _ in range(20):
                    flush.fill_(2)
                    g.replay()
            torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for k in range(steps):
            flush.fill_(k & 0xFF)
            starts[k].record(s)
            g.replay()
            ends[k].record(s)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = dist_max(sum(step_ms), world)
    return total_ms, step_ms


def single_call_us(rep: Replica, samples: int, world: int, T0: bool = False):
    """Median time of ONE call, from CUDA events around the replay of a graph that holds that
    call alone, L2 flushed before each sample (cold caches, launch latency included).  With
    T0, the same for a T = 0 call of the public API (one one-thread kernel that writes
    npp = 0): the floor that events, graph launch and one kernel launch cost by themselves."""
    import torch

    s = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    logits, bias, out = rep.sets[0]
    w = rep.w
    if T0:
        empty = torch.empty(0, w.E, dtype=torch.bfloat16, device="cuda")
        out0 = rep.mrs.RouteSortBuffers.allocate(0, w.E, w.topk, w.block_m, device="cuda")

    def call():
        if T0:
            rep.mrs.route_sort(empty, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                               w.block_m, out=out0, stream=s)
        else:
            rep.call(0, stream=s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(samples)]
    with torch.cuda.stream(s):
        for _ in range(3):
            flush.fill_(1)
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    with torch.cuda.stream(s):
        for k, (a, b) in enumerate(ev):
            flush.fill_(k & 0xFF)
            a.record(s)
            g.replay()
            b.record(s)
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3
    return dist_max(us, world)


def e2e_time(w, steps: int, warmup: int, world: int):
    """Whole calls through the public C ABI with host buffers: every step the host writes a
    fresh batch of logits into pinned host memory, and one moe_route_sort call reads it from
    there and writes every output into pinned host memory (both mapped into the device's
    address space with moe_route_sort_map_host: the transfers happen inside the call, over the
    host link, with no copies enqueued).  A ring of sets is reused only after a stream
    synchronisation (one per ring, inside the timed region).  CUDA events on the stream."""
    import torch

    import moe_expert_routing_sort_gb300 as mrs

    n_sets, n_batches = 32, 64
    src = [datagen.make_inputs(datagen.workload(w.name, seed=w.seed + i) if w.name in
                               datagen.WORKLOADS else w).logits_bf16 for i in range(n_batches)]
    bias = torch.from_numpy(datagen.make_inputs(w).bias).cuda()  # router parameter, resident
    h_logits = [torch.empty(w.T, w.E, dtype=torch.bfloat16, pin_memory=True)
                for _ in range(n_sets)]
    h_views = [t.view(torch.int16).numpy().view(np.uint16) for t in h_logits]
    outs = [mrs.RouteSortBuffers.allocate_pinned(w.T, w.E, w.topk, w.block_m)
            for _ in range(n_sets)]
    s = torch.cuda.Stream()
    lib = mrs.load()
    args = [(mrs.map_host(h_logits[i]), bias.data_ptr(), w.T, w.E, w.n_group, w.topk_group,
             w.topk, float(w.routed_scale), w.block_m, o.addr(o.topk_ids),
             o.addr(o.topk_weights), o.addr(o.sorted_token_ids), o.addr(o.sorted_weights),
             o.addr(o.expert_ids), o.addr(o.num_tokens_post_pad), o.workspace.data_ptr(),
             o.workspace.numel(), s.cuda_stream) for i, o in enumerate(outs)]

    def one(k):
        i = k % n_sets
        if i == 0 and k > 0:
            s.synchronize()  # every set's previous call has finished: the ring may be rewritten
        np.copyto(h_views[i], src[k % n_batches])  # this step's logits, written by the host
        rc = lib.moe_route_sort(*args[i])
        if rc != 0:
            raise RuntimeError(f"moe_route_sort: {mrs.strerror(rc)}")

    for k in range(max(warmup, n_sets)):
        one(k)
    s.synchronize()
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
    for k in range(steps):
        one(k)
    with torch.cuda.stream(s):
        b.record(s)
    torch.cuda.synchronize()
    barrier(world)
    ms = dist_max(a.elapsed_time(b), world)
    h2d = h_logits[0].numel() * 2
    d2h = outs[0].outputs.numel()
    return ms, h2d, d2h


def e2e_time_copies(w, steps: int, warmup: int, world: int):
    """The same end-to-end measurement where pinned host memory cannot be mapped: per step,
    one moe_route_sort_from_host call (copy of the host logits in, the call, one copy of the
    output block back), CUDA events on its stream."""
    import torch

    import moe_expert_routing_sort_gb300 as mrs

    inp = datagen.make_inputs(w)
    h_logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).pin_memory()
    bias = torch.from_numpy(inp.bias).cuda()
    d_logits = torch.empty_like(h_logits, device="cuda")
    out = mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m, device="cuda")
    h_out = torch.empty_like(out.outputs, device="cpu").pin_memory()
    s = torch.cuda.Stream()

    def one():
        mrs.route_sort_from_host(h_logits, d_logits, bias, w.n_group, w.topk_group, w.topk,
                                 w.routed_scale, w.block_m, out, h_out, stream=s)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
    for _ in range(steps):
        one()
    with torch.cuda.stream(s):
        b.record(s)
    torch.cuda.synchronize()
    barrier(world)
    return dist_max(a.elapsed_time(b), world), h_logits.numel() * 2, out.outputs.numel()


def n_sets_for(w) -> int:
    per = 2 * w.T * w.E
    return int(min(64, max(2, math.ceil(2 * L2_BYTES / max(per, 1)))))


def measure_workload(w, steps, warmup, world, peak_gbs, clocks=None):
    n_sets = n_sets_for(w) if w.T > 1 else 32
    rep = Replica(w, n_sets)
    total_ms, step_ms = time_graph_steps(rep, steps, warmup, world, clocks)
    calls = steps * n_sets
    # median over the timed steps (each step one graph of n_sets calls), slowest rank
    us_per_call = dist_max(statistics.median(step_ms), world) * 1e3 / n_sets
    npps = rep.npp()
    bytes_per_call = float(np.mean([algorithmic_bytes(w, n) for n in npps]))
    achieved = bytes_per_call / (us_per_call * 1e-6) / 1e9
    return {
        "us_per_call": us_per_call,
        "us_per_call_mean": total_ms * 1e3 / calls,
        "ms_per_step": total_ms / steps,
        "rep": rep,
        "calls_per_step": n_sets,
        "tokens_per_s": w.T / (us_per_call * 1e-6),
        "routes_per_s": w.T * w.topk / (us_per_call * 1e-6),
        "algorithmic_bytes_per_call": bytes_per_call,
        "achieved_gbs": achieved,
        "roofline_frac": achieved / peak_gbs,
        "launches": steps * n_sets * launches_per_call(w),
        "npp_mean": float(np.mean(npps)),
    }


def measure_sort_only(w, steps, warmup, world, atomic: bool, calls: int = 16):
    """moe_sort (deterministic) or moe_sort_atomic alone, on the routes route_sort gives for
    workload w: per-call time of a graph of `calls` calls, L2 flushed before each step."""
    import torch

    import moe_expert_routing_sort_gb300 as mrs

    inp = datagen.make_inputs(w)
    logits = torch.from_numpy(inp.logits_bf16.view(np.int16)).view(torch.bfloat16).cuda()
    bias = torch.from_numpy(inp.bias).cuda()
    routed = mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                            w.block_m)
    ids, wts = routed.topk_ids.clone(), routed.topk_weights.clone()
    outs = [mrs.RouteSortBuffers.allocate(w.T, w.E, w.topk, w.block_m) for _ in range(calls)]
    s = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def run():
        for o in outs:
            mrs.moe_sort(ids, wts, w.E, w.block_m, o.sorted_token_ids, o.sorted_weights,
                         o.expert_ids, o.num_tokens_post_pad, o.workspace, stream=s,
                         atomic=atomic)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    with torch.cuda.stream(s):
        for _ in range(warmup):
            flush.fill_(1)
            g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(world)
    with torch.cuda.stream(s):
        for k, (a, b) in enumerate(ev):
            flush.fill_(k & 0xFF)
            a.record(s)
            g.replay()
            b.record(s)
    torch.cuda.synchronize()
    ms = dist_max(sum(a.elapsed_time(b) for a, b in ev), world)
    return ms * 1e3 / (steps * calls)


def measure_gate(T, E, H, steps, warmup, world, peak_gbs, unfused=True):
    """moe_gate_route_sort (gate GEMV + the whole path) on the decode shape: per-call time of a
    graph over rotating sets (each its own gate matrix, more than twice the L2 in total, so
    every call reads its matrix from HBM), L2 flushed before each step.  With `unfused`, the
    same calls with the gate as a cuBLAS matmul followed by route_sort, for comparison."""
    import torch

    import moe_expert_routing_sort_gb300 as mrs

    w = datagen.workload(HEADLINE)
    n_sets = int(min(48, max(2, math.ceil(2 * L2_BYTES / (2 * E * H)))))
    sets = []
    for i in range(n_sets):
        inp = datagen.make_gate_inputs(T, E, H, seed=100 + i)
        hid = torch.from_numpy(inp.hidden_bf16.view(np.int16)).view(torch.bfloat16).cuda()
        wg = torch.from_numpy(inp.w_gate_bf16.view(np.int16)).view(torch.bfloat16).cuda()
        bias = torch.from_numpy(inp.bias).cuda()
        out = mrs.RouteSortBuffers.allocate(T, E, w.topk, w.block_m, device="cuda")
        logits = torch.empty(T, E, dtype=torch.bfloat16, device="cuda")
        sets.append((hid, wg, bias, out, logits))
    s = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def fused():
        for hid, wg, bias, out, logits in sets:
            mrs.gate_route_sort(hid, wg, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                                w.block_m, out=out, logits=logits, stream=s)

    def split():
        for hid, wg, bias, out, logits in sets:
            torch.matmul(hid, wg.t(), out=logits)
            mrs.route_sort(logits, bias, w.n_group, w.topk_group, w.topk, w.routed_scale,
                           w.block_m, out=out, stream=s)

    def per_call_us(fn):
        with torch.cuda.stream(s):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        with torch.cuda.stream(s):
            for _ in range(warmup):
                flush.fill_(1)
                g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        barrier(world)
        with torch.cuda.stream(s):
            for k, (a, b) in enumerate(ev):
                flush.fill_(k & 0xFF)
                a.record(s)
                g.replay()
                b.record(s)
        torch.cuda.synchronize()
        ms = dist_max(sum(a.elapsed_time(b) for a, b in ev), world)
        return ms * 1e3 / (steps * n_sets)

    us = per_call_us(fused)
    gate_bytes = 2 * E * H + 2 * T * H + 2 * T * E
    res = {"T": T, "E": E, "H": H, "us_per_call": us, "calls_per_step": n_sets,
           "gate_bytes_per_call": gate_bytes,
           "gate_bytes_over_whole_call_gbs": gate_bytes / (us * 1e-6) / 1e9,
           "gate_bytes_over_whole_call_frac": gate_bytes / (us * 1e-6) / 1e9 / peak_gbs,
           "launches_per_call": 2}
    if unfused:
        with torch.cuda.stream(s):
            split()  # cuBLAS picks its kernel outside capture
        res["unfused_cublas_gate_us_per_call"] = per_call_us(split)
    return res


# ----------------------------------------------------------------- CPU oracle
def cpu_oracle_rate(w, budget_s: float, runs: int = 5):
    """Time the oracle, pinned to one host core, on a bounded sample of workload w: the median
    of `runs` runs, each about budget_s / runs seconds.  Returns (seconds per token, sample)."""
    import oracle

    oracle.build()
    per_run = budget_s / runs
    with OneCore():
        if w.T == 1:
            inp = datagen.make_inputs(w)
            rates, total = [], 0
            for _ in range(runs):
                n = 0
                t0 = time.perf_counter()
                while time.perf_counter() - t0 < per_run:
                    oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group,
                                      w.topk, w.routed_scale, w.block_m)
                    n += 1
                rates.append((time.perf_counter() - t0) / n)
                total += n
            return statistics.median(rates), (f"median of {runs} runs, {total} whole calls on "
                                              f"the T=1 input ({budget_s:.0f} s), one core")
        # a token sample of the full workload: the whole path on the first n_tok tokens
        inp = datagen.make_inputs(w, T=min(w.T, 64))
        t0 = time.perf_counter()
        oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                          w.routed_scale, w.block_m)
        per_tok = (time.perf_counter() - t0) / inp.logits_bf16.shape[0]
        n_tok = int(max(16, min(w.T, per_run / max(per_tok, 1e-7))))
        inp = datagen.make_inputs(w, T=n_tok)
        rates = []
        for _ in range(runs):
            t0 = time.perf_counter()
            oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                              w.routed_scale, w.block_m)
            rates.append((time.perf_counter() - t0) / n_tok)
        return statistics.median(rates), (f"median of {runs} runs of the whole path on the "
                                          f"first {n_tok} of {w.T} tokens, one core")


def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle, as it stands, on this host (rank 0 only)."""
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    if w.T <= 64:
        inp = datagen.make_inputs(w)
        sample = f"the whole {w.name} call per step (T={w.T})"
    else:
        inp = datagen.make_inputs(w, T=64)
        sample = f"first 64 of {w.T} tokens per step, scaled to the full call"
    scale = w.T / inp.logits_bf16.shape[0]
    t_steps = []
    with OneCore():
        for k in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.route_sort(inp.logits_bf16, inp.bias, w.n_group, w.topk_group, w.topk,
                              w.routed_scale, w.block_m)
            el = (time.perf_counter() - t0) * scale
            if k >= args.warmup:
                t_steps.append(el)
    us = statistics.median(t_steps) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/call",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "E": w.E, "n_group": w.n_group,
                   "topk_group": w.topk_group, "topk": w.topk, "block_m": w.block_m,
                   "parallelism": "replicas" if world > 1 else "single"},
        "cpu_baseline": {"value": us, "unit": "us/call", "cores": 1, "kind": "oracle",
                         "sample": sample + " (median over steps, one core)",
                         "host": cpu_info()},
        "e2e": {"value": us, "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = datagen.workload(args.workload)
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch

    import moe_expert_routing_sort_gb300 as mrs

    mrs.load()  # fails loudly if the CUDA library is missing
    torch.cuda.set_device(local)
    peak, peak_kind = load_peaks()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local

    sampler = ClockSampler(gpu_index)
    sampler.start()
    head = measure_workload(w, args.steps, args.warmup, world, peak, clocks=True)
    clocks = sampler.stop()
    single = None
    if w.T <= 64:
        # one call alone (graph of one call, L2 flushed), beside the floor of a T = 0 call
        one = single_call_us(head["rep"], 200, world)
        floor = single_call_us(head["rep"], 200, world, T0=True)
        single = {"us": one, "t0_call_floor_us": floor, "us_above_floor": one - floor,
                  "how": "median of 200 samples: CUDA events around the replay of a graph "
                         "holding one call, L2 flushed before each; the floor is the same "
                         "measurement of a T=0 call (one one-thread kernel)"}
    try:
        e2e_ms, h2d, d2h = e2e_time(w, args.steps * 32, args.warmup, world)
        e2e_path = "zero-copy: pinned host logits and outputs mapped into the device space"
    except (mrs.RouteSortError, ValueError):  # host memory cannot be mapped on this system
        e2e_ms, h2d, d2h = e2e_time_copies(w, args.steps * 32, args.warmup, world)
        e2e_path = "copies: cudaMemcpyAsync in, the call, cudaMemcpyAsync out"
    e2e_us = e2e_ms * 1e3 / (args.steps * 32)

    configs = {}
    if not args.no_secondary:
        for name in SECONDARY:
            ws = datagen.workload(name)
            r = measure_workload(ws, max(3, min(args.steps, 10)), args.warmup, world, peak)
            configs[name] = {k: r[k] for k in ("us_per_call", "us_per_call_mean",
                                                 "tokens_per_s", "routes_per_s",
                                                 "achieved_gbs", "roofline_frac",
                                                 "algorithmic_bytes_per_call", "calls_per_step")}
            if ws.T > 1024:  # the sort step alone: deterministic order vs atomic slot order
                n = max(3, min(args.steps, 10))
                configs[name]["sort_only_us"] = {
                    "deterministic": measure_sort_only(ws, n, args.warmup, world, False),
                    "atomic_order": measure_sort_only(ws, n, args.warmup, world, True)}

    if not args.no_secondary:
        # per-call latency across token counts at the prefill shape (E = 896, G = 8, K = 16),
        # over the dispatch: one token, the single-CTA kernel, the per-token cooperative grid,
        # the warp-per-token cooperative grid and the three-kernel path
        sweep = {}
        for T in SWEEP_TOKENS:
            ws = datagen.workload("prefill_T512_E896", T=T)
            r = measure_workload(ws, max(3, min(args.steps, 10)), args.warmup, world, peak)
            sweep[str(T)] = r["us_per_call"]
        configs["prefill_E896_token_sweep"] = {"unit": "us/call", "us_per_call": sweep}

    if not args.no_secondary:
        # the router gate projection fused ahead of the path (batch-one decode shape)
        n = max(3, min(args.steps, 10))
        configs["gate_decode_T1_E896_H7168"] = measure_gate(1, 896, 7168, n, args.warmup,
                                                            world, peak)

    cpu = None
    if rank == 0:
        secs, sample = cpu_oracle_rate(w, args.cpu_budget)
        cpu = {"value": secs * 1e6, "unit": "us/call", "cores": 1, "kind": "oracle",
               "sample": sample, "host": cpu_info()}
        for name in configs:
            if name not in datagen.WORKLOADS:
                continue
            ws = datagen.workload(name)
            s2, samp2 = cpu_oracle_rate(ws, 3.0)
            configs[name]["cpu_oracle_tokens_per_s"] = 1.0 / s2
            configs[name]["cpu_oracle_sample"] = samp2

    if rank != 0:
        return 0
    # replicas: every rank makes its own calls, so the per-call latency is the slowest rank's;
    # the job's call rate is world times that rank's rate
    value = head["us_per_call"]
    traffic = captured_traffic(w.name)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "E": w.E, "n_group": w.n_group,
                   "topk_group": w.topk_group, "topk": w.topk, "block_m": w.block_m,
                   "routed_scale": w.routed_scale, "calls_per_step": head["calls_per_step"],
                   "l2": "flushed (256 MiB write) before every step; rotating input sets",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm",
                     "kernel": "mrs_decode_kernel (the whole call at T=1)" if w.T == 1 else
                               "moe_route_sort (whole call)",
                     "achieved": head["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": head["roofline_frac"], "peak_kind": peak_kind,
                     "traffic": traffic,
                     "traffic_source": ("profiles/dram_traffic.txt, capture of the current "
                                        "kernel sources " + kernel_source_hash())
                                       if traffic is not None else
                                       "no ncu capture of the current kernel sources"},
        "single_call": single,
        "job_calls_per_s": world * 1e6 / head["us_per_call"],
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "path": e2e_path},
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "configs": configs,
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
