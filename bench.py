#!/usr/bin/env python3
"""Benchmark of the depthwise causal conv1d decode update on GB300.

One step = one decode update (ccu_conv1d_update through the C-ABI) over the
large-batch decode workload: N=4096 rows, D=16384 channels, W=4, L=3, S=4096 slots,
BF16, bias, SiLU, slot indices a permutation with 5% padding rows. Inputs are seeded
and synthetic (the cuDNN page "Causal Conv1d Decode Update" publishes no dataset).

Metric: achieved HBM GB/s = algorithmic bytes / time, where the algorithmic bytes of
one update are, per active (row, channel): 2 B x read + 2L B state read + 2L B state
write + 2 B out write; per padding (row, channel): 2 B out write; plus weight, bias and
indices read once (1,026,899,968 B for this workload).

Printed: ONE JSON line (rank 0). ``value`` is device-resident throughput (inputs in
HBM, CUDA events on the launching stream); ``e2e`` adds, every step, the host->device
copy of that step's x and indices from pinned memory and the device->host copy of its
output; ``roofline`` reports the update kernel against the measured HBM copy peak;
``cpu_baseline`` times the single-threaded CPU oracle on a bounded sample;
``per_workload`` gives eager / CUDA-graph / cold-L2 µs per call for every workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) each rank runs its own copy of the workload on its own GPU
(independent decode batches: weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "conv1d_update HBM GB/s (% of GB300 peak) and µs/call vs N·D, 1 GPU"
try:
    PEAK_GBPS = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"])
except (OSError, KeyError, ValueError):
    PEAK_GBPS = 6800.0  # fallback figure when the measured peaks are absent
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
_CSRC = os.path.join(ROOT, "depthwise_causal_conv1d_gb300", "csrc")
# Per kernel family: the committed ncu summary of its DRAM traffic on the large-batch
# workload, and the sources whose hash that capture was taken with.
PROFILE_SUMMARIES = {
    "vector": (os.path.join(ROOT, "profiles", "update_vector_large_n4096_d16384.txt"),
               [os.path.join(_CSRC, f) for f in ("k_vector.cu", "ccu_vector.cuh", "ccu_internal.cuh")]),
    "bulk": (os.path.join(ROOT, "profiles", "update_bulk_large_n4096_d16384.txt"),
             [os.path.join(_CSRC, f) for f in ("k_bulk.cu", "ccu_bulk.cuh", "ccu_internal.cuh")]),
}


ALL_DECODE_WORKLOADS = {**synthetic.WORKLOADS, **synthetic.RING_WORKLOADS, **synthetic.WIDTH_WORKLOADS}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synthetic.BENCH_WORKLOAD, choices=sorted(ALL_DECODE_WORKLOADS),
                    help="a decode workload; the ring-buffer and width variants are for profiling rows of "
                         "the per-workload table")
    ap.add_argument("--rows", type=int, default=None,
                    help="run a smaller case of the same kernel: first ROWS rows (profiling)")
    ap.add_argument("--route", default="auto", choices=["auto", "scalar", "vector", "staged", "bulk"])
    ap.add_argument("--layout", default="compact", choices=["compact", "channel_last"])
    ap.add_argument("--quick", action="store_true",
                    help="device-resident timing only: no e2e, table, CPU baseline or clocks")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--table", choices=["prefill", "multi"], default=None,
                    help="time only the prefill or the multi-token rows, with --route, and print "
                         "them as one JSON line (profiling)")
    ap.add_argument("--table-reps", type=int, default=50, help="timed calls per row of --table")
    return ap.parse_args()


def workload_for(args) -> synthetic.Workload:
    wl = ALL_DECODE_WORKLOADS[args.workload]
    if args.rows is not None and args.rows < wl.N:
        changes = dict(N=args.rows)
        if wl.indices.startswith("perm"):
            changes["S"] = args.rows
        wl = synthetic.variant(wl, **changes)
    if args.layout != "compact":
        wl = synthetic.variant(wl, layout=args.layout)
    return wl


def config_of(wl: synthetic.Workload, extra=None) -> dict:
    cfg = {"workload": wl.name, "N": wl.N, "D": wl.D, "W": wl.W, "L": wl.L, "S": wl.S, "ld": wl.ld,
           "activation": wl.act, "bias": wl.has_bias, "indices": wl.indices, "pad_frac": wl.pad_frac,
           "state_layout": wl.layout, "N_x_D": wl.N * wl.D, "seed": wl.seed}
    if extra:
        cfg.update(extra)
    return cfg


# --------------------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local)
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

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        def parse(rows):
            out = []
            for _, ln in rows:
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 8:
                    continue
                try:
                    out.append(dict(sm=float(f[0]), smax=float(f[1]), reasons=f[4:8]))
                except ValueError:
                    continue
            return out

        inside = parse([r for r in self.lines if t0 <= r[0] <= t1])
        scope = "timed region"
        if not inside:
            inside = parse(self.lines)
            scope = "whole GPU phase (timed region shorter than one 200 ms sample)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = sorted({names[i] for s in inside for i, v in enumerate(s["reasons"]) if v == "Active"})
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["smax"] for s in inside), "reasons": seen,
                "samples": len(inside), "scope": scope}


def gpu_id_for(dev_index: int) -> str:
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        return parts[dev_index] if dev_index < len(parts) else str(dev_index)


# --------------------------------------------------------------------------- profile summary

def kernel_source_hash(route_name="vector") -> str:
    h = hashlib.sha256()
    for p in PROFILE_SUMMARIES[route_name][1]:
        with open(p, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(full_units: int, wl=None, route_name="vector"):
    """DRAM bytes per launch from the committed ncu summary of this kernel family, scaled to
    this launch's (row, channel) units; None if the kernel source changed since the capture,
    or if this run is not the captured kernel on the captured workload's kind of input."""
    if route_name not in PROFILE_SUMMARIES:
        return None, "no ncu capture for this route"
    if wl is not None:
        base = synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD]
        same_kind = (wl.D, wl.L, wl.W, wl.act, wl.layout, wl.ring) == (base.D, base.L, base.W, base.act,
                                                                    base.layout, base.ring)
        if not same_kind:
            return None, "no ncu capture for this workload"
    try:
        text = open(PROFILE_SUMMARIES[route_name][0]).read()
    except OSError:
        return None, "no ncu summary"
    kv = dict(ln.split("=", 1) for ln in text.splitlines() if "=" in ln and not ln.startswith("#"))
    try:
        if kv.get("kernel_source_sha256_16") != kernel_source_hash(route_name):
            return None, "kernel changed since the ncu capture"
        traffic = float(kv["dram_bytes_per_launch"])
        units = float(kv["units_per_launch"])
    except (KeyError, ValueError):
        return None, "ncu summary unreadable"
    return traffic * full_units / units, kv.get("capture_case", "")


# --------------------------------------------------------------------------- our arm

def to_dev(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


class Resident:
    """Device copies of one workload's tensors plus the C-ABI call on them."""

    def __init__(self, inp, dev, stream, route="auto", layout="compact"):
        import torch

        import depthwise_causal_conv1d_gb300 as ccu

        self.ccu = ccu
        wl = inp.wl
        self.wl = wl
        self.x_full = to_dev(inp.x, dev)
        self.x = self.x_full[:, :wl.D] if wl.ld != wl.D else self.x_full
        if layout == "compact":
            self.state = to_dev(inp.conv_state, dev)
        else:
            self.state = to_dev(synthetic.to_channel_last(inp.conv_state), dev).permute(0, 2, 1)
        self.w = to_dev(inp.weight, dev)
        self.b = to_dev(inp.bias, dev) if inp.bias is not None else None
        self.idx = torch.from_numpy(inp.indices).to(dev) if inp.indices is not None else None
        self.idx_host = inp.indices
        self.seq = (torch.from_numpy(inp.cache_seqlens).to(dev) if inp.cache_seqlens is not None
                    else None)
        self.out = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, device=dev)
        self.stream = stream
        self.route = ccu.ROUTES[route]
        ss, sd, sl = self.state.stride()
        self.args = (self.x.data_ptr(), wl.ld, self.state.data_ptr(), ss, sd, sl, self.w.data_ptr(),
                     None if self.b is None else self.b.data_ptr(),
                     ccu.CCU_ACT_SILU if wl.act == "silu" else ccu.CCU_ACT_IDENTITY,
                     None if self.idx is None else self.idx.data_ptr(),
                     None if self.seq is None else self.seq.data_ptr(),
                     wl.N, wl.D, wl.S, wl.L, wl.W, self.out.data_ptr(), None, self.route,
                     stream.cuda_stream)
        st, chosen = ccu.ccu_conv1d_select_route(*self.args[:17], self.route)
        ccu.raise_for_status(st)
        self.route_name = ccu.ccu_route_name(chosen)

    def call(self):
        st = self.ccu.lib.ccu_conv1d_update_ex(*self.args)
        if st != 0:
            self.ccu.raise_for_status(st)

    def rotating_args(self, k):
        """Argument tuples of k calls, each on its own device copies of x, conv_state and out
        (weights, bias, indices and cache_seqlens are shared: they are read, not written)."""
        import torch

        self.copies = [(self.x_full.clone(), self.state.clone(), torch.empty_like(self.out)) for _ in range(k)]
        torch.cuda.synchronize()  # the copies are made on the current stream; the calls run on another
        out = []
        for xf, st, o in self.copies:
            a = list(self.args)
            a[0], a[2], a[16] = xf.data_ptr(), st.data_ptr(), o.data_ptr()
            out.append(tuple(a))
        return out


def time_device_resident(res: Resident, steps: int, warmup: int, world: int, dev):
    """Back-to-back calls on one stream, two CUDA events around the timed region.

    Returns (seconds for the K steps, max over ranks; mean seconds per launch; wall times).
    """
    import torch

    s = res.stream
    for _ in range(warmup):
        res.call()
    torch.cuda.synchronize()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_begin.record(s)
    for _ in range(steps):
        res.call()
    t_end.record(s)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    local = t_begin.elapsed_time(t_end) / 1e3
    total = max_over_ranks(local, world, dev)
    return total, local / steps, (wall0, wall1)


def time_e2e_pipelined(res: Resident, inp, steps: int, warmup: int, world: int, dev, chunks: int = 8):
    """End to end with copy-engine transfers around the C-ABI call.

    Every step copies that step's x and indices from pinned host memory to the device,
    runs the update, and copies the output back to pinned host memory. A step is split
    into row chunks on three streams (host->device, update, device->host) so the copies of
    one chunk overlap the update of another; device x/indices/out are double-buffered by
    step parity so consecutive steps can overlap too. The update of chunk i of step k
    waits for its own input copy, and its output copy waits for the update.
    """
    import torch

    wl = inp.wl
    ccu = res.ccu
    N = wl.N
    h_x = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp.indices).pin_memory() if inp.indices is not None else None
    h_out = torch.empty((N, wl.D), dtype=torch.bfloat16, pin_memory=True)
    bytes_in = h_x.numel() * 2 + (h_idx.numel() * 4 if h_idx is not None else 0)
    bytes_out = h_out.numel() * 2
    d_x = [res.x_full, torch.empty_like(res.x_full)]
    d_idx = [res.idx, torch.empty_like(res.idx)] if res.idx is not None else [None, None]
    d_out = [res.out, torch.empty_like(res.out)]
    s_in, s_k, s_out = torch.cuda.Stream(dev), res.stream, torch.cuda.Stream(dev)
    bounds = [(N * i // chunks, N * (i + 1) // chunks) for i in range(chunks)]
    ev_in = [[torch.cuda.Event() for _ in range(chunks)] for _ in range(2)]
    ev_k = [[torch.cuda.Event() for _ in range(chunks)] for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(chunks)] for _ in range(2)]
    used = [False, False]
    base = list(res.args)
    act, ld = base[8], base[1]

    def step(k):
        b = k & 1
        for i, (r0, r1) in enumerate(bounds):
            if r1 == r0:
                continue
            with torch.cuda.stream(s_in):
                if used[b]:
                    s_in.wait_event(ev_k[b][i])  # the previous user of this buffer has read it
                d_x[b][r0:r1].copy_(h_x[r0:r1], non_blocking=True)
                if h_idx is not None:
                    d_idx[b][r0:r1].copy_(h_idx[r0:r1], non_blocking=True)
                ev_in[b][i].record(s_in)
            s_k.wait_event(ev_in[b][i])
            if used[b]:
                s_k.wait_event(ev_out[b][i])  # its earlier output has left the device
            xv = d_x[b][r0:r1, :wl.D]
            st = ccu.lib.ccu_conv1d_update(
                xv.data_ptr(), ld, base[2], base[3], base[4], base[5], base[6], base[7], act,
                None if d_idx[b] is None else d_idx[b][r0:r1].data_ptr(), None, r1 - r0, wl.D,
                wl.S, wl.L, wl.W, d_out[b][r0:r1].data_ptr(), s_k.cuda_stream)
            if st != 0:
                ccu.raise_for_status(st)
            ev_k[b][i].record(s_k)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[b][i])
                h_out[r0:r1].copy_(d_out[b][r0:r1], non_blocking=True)
                ev_out[b][i].record(s_out)
        used[b] = True

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_in)
    s_k.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(steps):
        step(warmup + k)
    s_in.wait_stream(s_k)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    barrier(world)
    total = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    # copy rates alone, for context
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c2 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_in):
        c0.record(s_in)
        d_x[0].copy_(h_x, non_blocking=True)
        c1.record(s_in)
        h_out.copy_(d_out[0], non_blocking=True)
        c2.record(s_in)
    torch.cuda.synchronize()
    rates = {"h2d_GBps_alone": round(h_x.numel() * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9, 1),
             "d2h_GBps_alone": round(bytes_out / (c1.elapsed_time(c2) * 1e-3) / 1e9, 1)}
    # Both directions at once (x in on one stream, out back on another): the copy engines'
    # two-way rate over the host link for a step's traffic. Best of three.
    best = None
    for _ in range(3):
        c3, c4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c3.record(s_in)
        s_out.wait_event(c3)
        with torch.cuda.stream(s_in):
            d_x[0].copy_(h_x, non_blocking=True)
        with torch.cuda.stream(s_out):
            h_out.copy_(d_out[0], non_blocking=True)
        s_in.wait_stream(s_out)
        c4.record(s_in)
        torch.cuda.synchronize()
        sec = c3.elapsed_time(c4) * 1e-3
        best = sec if best is None else min(best, sec)
    rates["bidir_GBps"] = round((h_x.numel() * 2 + bytes_out) / best / 1e9, 1)
    return total, bytes_in, bytes_out, rates, chunks


def time_e2e_zero_copy(res: Resident, inp, steps: int, warmup: int, world: int, dev):
    """End to end through the C-ABI with host buffers.

    Every step calls ccu_conv1d_update with x and out in pinned host memory (allocated
    with cudaHostAlloc by torch, so the device addresses them directly under unified
    addressing): the kernel reads the step's x from the host and writes its output to the
    host over the host link, with no staging copy; the step's indices are copied
    host->device first. conv_state and the weights stay resident in HBM.
    """
    import torch

    wl = inp.wl
    ccu = res.ccu
    h_x = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp.indices).pin_memory() if inp.indices is not None else None
    h_out = torch.empty((wl.N, wl.D), dtype=torch.bfloat16, pin_memory=True)
    bytes_in = h_x.numel() * 2 + (h_idx.numel() * 4 if h_idx is not None else 0)
    bytes_out = h_out.numel() * 2
    s = res.stream
    base = list(res.args)

    def step():
        if h_idx is not None:
            with torch.cuda.stream(s):
                res.idx.copy_(h_idx, non_blocking=True)
        st = ccu.lib.ccu_conv1d_update(h_x.data_ptr(), base[1], base[2], base[3], base[4], base[5],
                                       base[6], base[7], base[8], base[9], None, wl.N, wl.D, wl.S,
                                       wl.L, wl.W, h_out.data_ptr(), s.cuda_stream)
        if st != 0:
            ccu.raise_for_status(st)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s)
    for _ in range(steps):
        step()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    total = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    return total, bytes_in, bytes_out


def cold_rotating_us(res, stream, passes=3):
    """µs per call with nothing of the call's own data in L2: K back-to-back calls, each on its
    own copies of x, conv_state and out, the K copies together at least 3x the L2 (each
    copy was last touched K - 1 calls earlier); two CUDA events around each pass of K
    calls, the median pass divided by K. One call between two events cannot resolve a few
    microseconds (the events tick in ~2 µs steps on this GPU)."""
    import torch

    wl = res.wl
    touched = synthetic.algorithmic_bytes(wl, res.idx_host)
    k = max(4, -(-3 * L2_BYTES // max(touched, 1)))
    args = res.rotating_args(k)
    lib = res.ccu.lib

    def one_pass():
        for a in args:
            st = lib.ccu_conv1d_update_ex(*a)
            if st != 0:
                res.ccu.raise_for_status(st)

    one_pass()
    torch.cuda.synchronize()
    per = []
    for _ in range(passes):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one_pass()
        e1.record(stream)
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) * 1e3 / k)
    res.copies = None
    return statistics.median(per), k


def per_workload_table(dev, stream, reps=50):
    """µs per call for every decode workload: eager (back to back on the same buffers, so a
    workload smaller than L2 is served from it), CUDA-graph replay, and cold (back-to-back
    calls on rotating copies larger than L2 together, see cold_rotating_us). The roofline
    fraction of a workload that fits in L2 comes from its cold time."""
    import torch

    rows = {}
    for name, wl in {**synthetic.WORKLOADS, **synthetic.RING_WORKLOADS,
                     **synthetic.WIDTH_WORKLOADS}.items():
        inp = synthetic.generate(wl)
        res = Resident(inp, dev, stream, layout=wl.layout)
        nbytes = synthetic.algorithmic_bytes(wl, inp.indices)
        for _ in range(5):
            res.call()
        torch.cuda.synchronize()
        # eager, back to back
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            res.call()
        b.record(stream)
        torch.cuda.synchronize()
        eager_us = a.elapsed_time(b) * 1e3 / reps
        cold_us, k = cold_rotating_us(res, stream)
        # CUDA graph: 100 calls captured, replayed 20 times
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(100):
                res.call()
        with torch.cuda.stream(stream):  # replay on the stream the events are recorded on
            g.replay()
            torch.cuda.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(20):
                g.replay()
            g1.record(stream)
        torch.cuda.synchronize()
        graph_us = g0.elapsed_time(g1) * 1e3 / 2000
        rows[name] = {"N_x_D": wl.N * wl.D, "bytes": nbytes, "route": res.route_name,
                      "state": f"{'ring' if wl.ring else 'linear'} {wl.layout}", "W": wl.W, "L": wl.L,
                      "eager_us": round(eager_us, 3), "graph_us": round(graph_us, 3),
                      "cold_us": round(cold_us, 3), "cold_copies": k,
                      "cold_GBps": round(nbytes / (cold_us * 1e-6) / 1e9, 1),
                      "cold_frac": round(nbytes / (cold_us * 1e-6) / 1e9 / PEAK_GBPS, 4),
                      "warm_frac": round(nbytes / (eager_us * 1e-6) / 1e9 / PEAK_GBPS, 4)}
        del g, res
    return rows


def n_curve(dev, stream, reps=100):
    """µs per call against N·D: the large-batch decode settings (D=16384, L=3, SiLU, bias,
    permuted slots with 5% padding) at N = 1, 8, 64, 256, 1024, 4096, route AUTO; warm
    (back to back on the same buffers) and cold (rotating copies, see cold_rotating_us)."""
    import torch

    base = synthetic.WORKLOADS[synthetic.BENCH_WORKLOAD]
    rows = {}
    for n in (1, 8, 64, 256, 1024, 4096):
        wl = synthetic.variant(base, N=n, S=n)
        inp = synthetic.generate(wl)
        res = Resident(inp, dev, stream)
        nbytes = synthetic.algorithmic_bytes(wl, inp.indices)
        for _ in range(5):
            res.call()
        torch.cuda.synchronize()
        k = max(20, min(reps * 10, int(2e10 / max(nbytes, 1))))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            res.call()
        b.record(stream)
        torch.cuda.synchronize()
        warm_us = a.elapsed_time(b) * 1e3 / k
        cold_us, copies = cold_rotating_us(res, stream)
        rows[f"N={n}"] = {"N_x_D": wl.N * wl.D, "bytes": nbytes, "route": res.route_name,
                          "warm_us": round(warm_us, 3), "cold_us": round(cold_us, 3), "cold_copies": copies,
                          "cold_GBps": round(nbytes / (cold_us * 1e-6) / 1e9, 1),
                          "cold_frac": round(nbytes / (cold_us * 1e-6) / 1e9 / PEAK_GBPS, 4)}
        del res
    return rows


def checked_cost_rows(dev, stream, reps=100):
    """µs per call, back to back, of the update unchecked, range-checked
    (ccu_conv1d_update_checked) and range- and duplicate-checked in the same launch
    (ccu_conv1d_update_checked_ex with its slot scratch cleared by the call), on the paged
    (N=256, D=8192, S=1024) and the large-batch workloads, AUTO route."""
    import torch

    rows = {}
    for name in ("paged_n256_d8192_l3_s1024_pad10_silu", synthetic.BENCH_WORKLOAD):
        wl = synthetic.WORKLOADS[name]
        inp = synthetic.generate(wl)
        res = Resident(inp, dev, stream)
        lib = res.ccu.lib
        status = torch.zeros((1,), dtype=torch.int32, device=dev)
        scratch = torch.zeros((wl.S,), dtype=torch.int32, device=dev)
        a = list(res.args)
        a[18] = 0  # AUTO
        plain = tuple(a)
        a[17] = status.data_ptr()
        checked = tuple(a)
        ex = tuple(a[:18]) + (scratch.data_ptr(),) + tuple(a[18:])
        calls = {"unchecked": lambda: lib.ccu_conv1d_update_ex(*plain),
                 "range_checked": lambda: lib.ccu_conv1d_update_ex(*checked),
                 "range_and_duplicate_checked": lambda: lib.ccu_conv1d_update_checked_ex(*ex)}
        row = {"N_x_D": wl.N * wl.D, "route": res.route_name}
        for label, fn in calls.items():
            for _ in range(5):
                st = fn()
                if st != 0:
                    res.ccu.raise_for_status(st)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            row[f"{label}_us"] = round(e0.elapsed_time(e1) * 1e3 / reps, 3)
        row["status"] = int(status.item())
        rows[name] = row
        del res
    return rows


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def multi_token_rows(dev, stream, reps=50, route=0, singles_too=True):
    """µs per call of the multi-token update, and of the same tokens as T single calls."""
    import torch

    import depthwise_causal_conv1d_gb300 as ccu

    rows = {}
    for name, wl in synthetic.MULTI_WORKLOADS.items():
        inp = synthetic.generate(wl)
        N, D, T, L = wl.N, wl.D, wl.T, wl.L
        x = to_dev(inp.x, dev)  # [N, T, D] memory
        st = to_dev(inp.conv_state, dev)
        w, b = to_dev(inp.weight, dev), to_dev(inp.bias, dev)
        idx = torch.from_numpy(inp.indices).to(dev)
        seq = torch.from_numpy(inp.cache_seqlens).to(dev) if inp.cache_seqlens is not None else None
        seq_ptr = None if seq is None else seq.data_ptr()
        out = torch.empty((N, T, D), dtype=torch.bfloat16, device=dev)
        out1 = torch.empty((N, D), dtype=torch.bfloat16, device=dev)  # one token's output
        act = ccu.CCU_ACT_SILU if wl.act == "silu" else ccu.CCU_ACT_IDENTITY

        def multi():
            stat = ccu.lib.ccu_conv1d_update_multi(
                x.data_ptr(), T * D, 1, D, st.data_ptr(), D * L, L, 1, w.data_ptr(), b.data_ptr(), act,
                idx.data_ptr(), seq_ptr, N, D, T, wl.S, L, wl.W, out.data_ptr(), T * D, 1, D, None, None,
                route, stream.cuda_stream)
            if stat != 0:
                ccu.raise_for_status(stat)

        def singles():
            # a ring state advances one entry per token: the token's position comes from
            # cache_seqlens + t (the counts a caller would pass), here precomputed per token
            for t in range(T):
                stat = ccu.lib.ccu_conv1d_update(
                    x[:, t].data_ptr(), T * D, st.data_ptr(), D * L, L, 1, w.data_ptr(), b.data_ptr(),
                    act, idx.data_ptr(), None if seq is None else seqs[t].data_ptr(), N, D, wl.S, L, wl.W,
                    out1.data_ptr(), stream.cuda_stream)
                if stat != 0:
                    ccu.raise_for_status(stat)

        seqs = [seq + t for t in range(T)] if seq is not None else None

        res = {}
        for label, fn in (("multi", multi), ("singles", singles))[:2 if singles_too else 1]:
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            e.record(stream)
            torch.cuda.synchronize()
            res[label] = a.elapsed_time(e) * 1e3 / reps
        nbytes = synthetic.algorithmic_bytes(wl, inp.indices)
        rows[name] = {"N_x_D": N * D, "T": T, "bytes": nbytes, "us_per_call": round(res["multi"], 3),
                      "GBps": round(nbytes / (res["multi"] * 1e-6) / 1e9, 1),
                      "frac": round(nbytes / (res["multi"] * 1e-6) / 1e9 / PEAK_GBPS, 4),
                      "same_tokens_as_T_single_calls_us": round(res.get("singles", float("nan")), 3)}
    return rows


def prefill_rows(dev, stream, reps=50, route=0):
    """µs per call of the full-sequence prefill (with its channel-last final state)."""
    import torch

    import depthwise_causal_conv1d_gb300 as ccu

    rows = {}
    for name, spec in synthetic.PREFILL_WORKLOADS.items():
        x_btd, weight, bias = synthetic.generate_prefill(spec)
        B, T, D, L = spec["B"], spec["T"], spec["D"], spec["L"]
        x = to_dev(x_btd, dev).permute(0, 2, 1)  # [B, D, T] view of token-major memory
        w = to_dev(weight, dev)
        b = to_dev(bias, dev) if bias is not None else None
        out = torch.empty_like(x)
        fin = torch.empty((B, L, D), dtype=torch.bfloat16, device=dev).permute(0, 2, 1)
        act = ccu.CCU_ACT_SILU if spec["act"] == "silu" else ccu.CCU_ACT_IDENTITY

        def call():
            st = ccu.lib.ccu_causal_conv1d_fwd(
                x.data_ptr(), *x.stride(), w.data_ptr(), None if b is None else b.data_ptr(), act,
                None, 0, 0, 0, B, D, T, L, spec["W"], out.data_ptr(), *out.stride(), fin.data_ptr(),
                *fin.stride(), route, stream.cuda_stream)
            if st != 0:
                ccu.raise_for_status(st)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call()
        e.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(e) * 1e3 / reps
        nbytes = synthetic.prefill_bytes(spec)
        rows[name] = {"B_x_T_x_D": B * T * D, "bytes": nbytes, "us_per_call": round(us, 3),
                      "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                      "frac": round(nbytes / (us * 1e-6) / 1e9 / PEAK_GBPS, 4)}
    return rows


def cpu_baseline_sample(inp, target_s: float):
    """Time the single-threaded C oracle on a bounded sample of the workload's rows."""
    import oracle

    wl = inp.wl
    lib = oracle.load()
    # first a small probe to size the sample
    rows = max(1, min(wl.N, 64))
    t_probe = _oracle_rows(oracle, lib, inp, rows)
    per_row = t_probe / rows
    rows = int(max(1, min(wl.N, (target_s / 3) / max(per_row, 1e-9))))
    times = [_oracle_rows(oracle, lib, inp, rows) for _ in range(3)]
    t = statistics.median(times)
    sub_idx = inp.indices[:rows] if inp.indices is not None else None
    sub_wl = synthetic.variant(wl, N=rows)
    nbytes = synthetic.algorithmic_bytes(sub_wl, sub_idx)
    return {"value": round(nbytes / t / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {wl.N} rows (all {wl.D} channels, full state), "
                      f"median of 3 runs of {t:.2f} s each; {nbytes} algorithmic bytes per run",
            "seconds_per_run": round(t, 3), "cores_available": os.cpu_count(), "cpu_model": cpu_model()}


def _oracle_rows(oracle, lib, inp, rows):
    wl = inp.wl
    state = inp.conv_state.copy()  # outside the timed region
    x = np.ascontiguousarray(inp.x[:rows])
    idx = inp.indices[:rows].copy() if inp.indices is not None else None
    t0 = time.perf_counter()
    oracle.conv1d_update(x, wl.ld, state, (wl.D * wl.L, wl.L, 1), inp.weight, inp.bias, wl.act,
                         idx, rows, wl.D, wl.S, wl.L, wl.W, lib=lib)
    return time.perf_counter() - t0


def run_ours(args):
    import torch

    world, rank, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = workload_for(args)
    inp = synthetic.generate(wl)
    nbytes = synthetic.algorithmic_bytes(wl, inp.indices)
    stream = torch.cuda.Stream(device=dev)
    res = Resident(inp, dev, stream, route=args.route, layout=wl.layout)

    sampler = None
    if not args.quick:
        sampler = ClockSampler(gpu_id_for(local))
        sampler.start()
        time.sleep(0.3)

    total, per_launch, (w0, w1) = time_device_resident(res, args.steps, args.warmup, world, dev)
    value = nbytes * world * args.steps / total / 1e9
    achieved = nbytes / per_launch / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 6800.0, "fallback"
    traffic, traffic_note = ncu_traffic(wl.N * wl.D, wl, res.route_name)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; the pages publish no dataset)",
        "config": config_of(wl, {"route": res.route_name,
                                 "l2": f"inputs larger than L2: {nbytes / 1e9:.3f} GB touched per "
                                       f"step vs {L2_BYTES / 2**20:.0f} MiB L2",
                                 "us_per_call": round(total / args.steps * 1e6, 2),
                                 "parallelism": f"independent decode batch per GPU x{world}"}),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (hbm_gbs)",
                     "bytes_per_launch": nbytes,
                     "launch_us": round(per_launch * 1e6, 2),
                     "launch_timing": "CUDA events around the K back-to-back launches on their stream",
                     "frac_of_nominal_8TBps": round(achieved / 8000.0, 4),
                     "traffic": None if traffic is None else round(traffic),
                     "traffic_note": traffic_note},
        "gpu_launches": args.steps,
    }
    if not args.quick:
        e2e_steps = max(10, min(200, args.steps // 20))
        e2e_total, bi, bo = time_e2e_zero_copy(res, inp, e2e_steps, 3, world, dev)
        pipe_total, _, _, rates, nchunks = time_e2e_pipelined(res, inp, e2e_steps, 3, world, dev)
        line["e2e"] = {"value": round(nbytes * world * e2e_steps / e2e_total / 1e9, 1), "unit": UNIT,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "ms_per_step": round(e2e_total / e2e_steps * 1e3, 4), "steps": e2e_steps,
                       "path": "ccu_conv1d_update on pinned host x and out (the kernel reads x from and "
                               "writes out to host memory over the host link); indices copied "
                               "host->device each step; conv_state and weights resident in HBM",
                       "copy_engine_pipeline": {
                           "value": round(nbytes * world * e2e_steps / pipe_total / 1e9, 1),
                           "ms_per_step": round(pipe_total / e2e_steps * 1e3, 4),
                           "path": f"x/indices copied host->device and out device->host by copy "
                                   f"engines, {nchunks} row chunks on three streams", **rates}}
        # The step's host traffic at the copy engines' two-way rate: frac near or above 1
        # means the e2e path is bound by the host link, not by the kernel.
        link_ms = (bi + bo) / (rates["bidir_GBps"] * 1e9) * 1e3
        line["e2e"]["host_link"] = {
            "bidir_GBps": rates["bidir_GBps"], "step_ms_at_copy_engine_rate": round(link_ms, 4),
            "frac": round(link_ms / (e2e_total / e2e_steps * 1e3), 3),
            "note": "x in and out back as two concurrent copy-engine transfers of the whole step; "
                    "the kernel's own loads and stores from pinned memory may beat it (frac > 1)"}
        sampler.stop()
        line["clocks"] = sampler.summary(w0, w1)
        if rank == 0 and world == 1:
            line["per_workload"] = per_workload_table(dev, stream)
            line["n_curve"] = n_curve(dev, stream)
            line["multi_token"] = multi_token_rows(dev, stream)
            line["prefill"] = prefill_rows(dev, stream)
            line["checked_cost"] = checked_cost_rows(dev, stream)
        if rank == 0:
            line["cpu_baseline"] = cpu_baseline_sample(inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_table(args):
    """Only the prefill or the multi-token rows (one JSON line); for profiling one kernel."""
    import torch

    import depthwise_causal_conv1d_gb300 as ccu

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    route = ccu.ROUTES[args.route]
    if args.table == "prefill":
        rows = prefill_rows(dev, stream, args.table_reps, route)
    else:
        rows = multi_token_rows(dev, stream, args.table_reps, route, singles_too=False)
    print(json.dumps({"table": args.table, "route": args.route, "reps": args.table_reps, "rows": rows}),
          flush=True)


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores (rank 0 only)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    wl = workload_for(args)
    inp = synthetic.generate(wl)
    lib = oracle.load()
    # each step: a bounded sample of the workload's rows, sized so the run takes minutes
    probe = _oracle_rows(oracle, lib, inp, min(wl.N, 16)) / min(wl.N, 16)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.N, budget / max(probe, 1e-9))))
    for _ in range(args.warmup):
        _oracle_rows(oracle, lib, inp, rows)
    times = [_oracle_rows(oracle, lib, inp, rows) for _ in range(args.steps)]
    total = sum(times)
    sub_wl = synthetic.variant(wl, N=rows)
    nbytes = synthetic.algorithmic_bytes(sub_wl, inp.indices[:rows] if inp.indices is not None else None)
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; the pages publish no dataset)",
        "config": config_of(wl),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {rows} of {wl.N} rows per step (all {wl.D} channels)",
                         "rows_per_step": rows,
                         "cores_available": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3  # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.table is not None:
        run_table(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
