#!/usr/bin/env python
"""Throughput of exact fused attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole path over one batch of the workload: the
forward (one launch) and, for workloads with a backward, the backward's three
launches (preprocess, fused dK/dV/dQ, dQ convert), all through the C ABI.
FLOPs per step use the library's formula: 4 B H N^2 d for the forward, halved
under the causal mask, and 2.5 times that for the backward.

Prints ONE JSON line (rank 0).  ``value`` is device-timed TFLOP/s over all
ranks with inputs resident in HBM; ``e2e`` is the same metric through the
same C ABI with pinned host buffers copied in and results copied out inside
the timed region; ``roofline`` reports the dominant kernel against the
measured bf16 peak; ``cpu_baseline`` times the fp64 CPU oracle on a bounded
sample.  Under torchrun each rank runs an independent replica of the
workload on its own GPU (no collective on the data path; weak scaling).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s and % of GB300 dense BF16 peak (1 GPU)"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "exact_io_aware_31_gb300", "csrc")


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer twice the L2's size, then
    reads another one as large, so the written lines are back in HBM before
    the next timed step instead of being written back during it."""

    def __init__(self, device):
        self.w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def flops_per_step(w):
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        f /= 2
    fwd = f
    bwd = 2.5 * f if w.backward else 0.0
    return fwd, bwd


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device):
    """Largest value of ``x`` over all ranks (``x`` itself when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Throughput of all ranks together: every rank runs one replica step in ``ms_per_step``."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


# The translation unit of each profiled kernel; its hash covers that file and
# every header it includes (followed through #include, as the build does).
KERNEL_SOURCES = {
    "fa_fwd_kernel": "fa_fwd.cu",
    "fa_fwd_kernel_fp8": "fa_fwd.cu",
    "fa_bwd_pre": "fa_bwd.cu",
    "fa_bwd_main": "fa_bwd.cu",
    "fa_bwd_dq_conv": "fa_bwd.cu",
}


def source_hash(kernel):
    from exact_io_aware_31_gb300 import build
    h = hashlib.sha256()
    for path in build.build_inputs(CSRC, (KERNEL_SOURCES[kernel],)):
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + f.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, workload):
    """Bytes per launch from a committed ncu capture, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    rec = table.get(kernel, {}).get(workload)
    if not rec or kernel not in KERNEL_SOURCES or rec.get("source_sha") != source_hash(kernel):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sms.append(float(parts[0]))
                    maxes.append(float(parts[1]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[3:7]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "samples": len(sms),
                "reasons": sorted(reasons)}


ORACLE_ROWS = 1024  # query rows per oracle sample unit


def oracle_units(w):
    """Sample units of the workload for the CPU oracle: (slice b, slice h, first row, rows).

    A unit is one block of up to ORACLE_ROWS query rows of one (b, h) slice,
    forward and (for workloads with a backward) that block's whole share of
    the backward: its dQ rows and its terms of dK and dV.  Units are visited
    spread over slices and row blocks, in a fixed order."""
    nblk = (w.N + ORACLE_ROWS - 1) // ORACLE_ROWS
    units = []
    for i in range(w.B * w.H * nblk):
        sl = i % (w.B * w.H)
        blk = (i // (w.B * w.H) + 7 * sl) % nblk
        b, h = divmod(sl, w.H)
        r0 = blk * ORACLE_ROWS
        units.append((b, h, r0, min(ORACLE_ROWS, w.N - r0)))
    return units


def oracle_unit_flops(w, r0, rows):
    """The metric's FLOPs (fwd + bwd) carried by query rows r0 .. r0 + rows - 1 of one slice.

    A slice's FLOPs are shared out in proportion to the (query, key) pairs each
    row covers: all N keys, or under the causal mask keys 0 .. i for row i,
    so a sample of early (light) and late (heavy) row blocks is credited
    with the work it really did."""
    fwd, bwd = flops_per_step(w)
    per_slice = (fwd + bwd) / (w.B * w.H)
    if not w.causal:
        return per_slice * rows / w.N
    pairs = rows * r0 + rows * (rows + 1) // 2  # sum of (i + 1) over the rows
    return per_slice * pairs / (w.N * (w.N + 1) // 2)


def oracle_run_unit(w, q, k, v, do, unit):
    import oracle
    b, h, r0, rows = unit
    qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
    if w.backward:
        oracle.attention_backward_head_rows(qd, kd, vd, dod, range(r0, r0 + rows), w.scale, w.causal)
    else:
        oracle.attention_forward_head_rows(qd, kd, vd, range(r0, r0 + rows), w.scale, w.causal)


def oracle_sample(w, q, k, v, do, seconds, start=0):
    """Time the fp64 oracle on sample units (at least one) for about `seconds`: (TFLOP/s, units, s)."""
    units = oracle_units(w)
    done, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        unit = units[(start + done) % len(units)]
        oracle_run_unit(w, q, k, v, do, unit)
        flops += oracle_unit_flops(w, unit[2], unit[3])
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return flops / el / 1e12, done, el


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, w):
    """The fp64 CPU oracle on the host cores; each step is one bounded sample unit of the workload.

    ``ms_per_step`` is the measured mean time of those sampled steps;
    ``extrapolated_ms_per_workload_step`` scales it to the whole workload by
    the metric's FLOPs and is not a measurement."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    q, k, v, do = workloads.workload_inputs(w)
    units = oracle_units(w)
    times, flops = [], []
    for i in range(args.warmup + args.steps):
        unit = units[i % len(units)]
        t0 = time.perf_counter()
        oracle_run_unit(w, q, k, v, do, unit)
        el = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(el)
            flops.append(oracle_unit_flops(w, unit[2], unit[3]))
    value = sum(flops) / sum(times) / 1e12
    fwd, bwd = flops_per_step(w)
    ms = 1e3 * sum(times) / len(times)
    sample = (f"each step one unit of up to {ORACLE_ROWS} query rows of one (b,h) slice (fwd"
              f"{' + its whole share of the bwd' if w.backward else ''}) in fp64 numpy, units spread over "
              f"slices and row blocks; {len(times)} timed steps, {sum(times):.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "extrapolated_ms_per_workload_step": round(1e3 * (fwd + bwd) / (value * 1e12), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**w.describe(), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import exact_io_aware_31_gb300 as fa
    from exact_io_aware_31_gb300 import build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    fa.load_library()

    q, k, v, do = workloads.workload_inputs(w, rank=rank)  # each rank: its own batch
    B, H, N, d = w.B, w.H, w.N, w.d
    dev = torch.device("cuda", local)
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qg)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(qg) for _ in range(3))
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    scale, causal = w.scale, int(w.causal)
    in_bytes = qg.numel() * 2
    flush = in_bytes < L2_BYTES
    flush_l2 = L2Flush(dev) if flush else None

    def check(st, where):
        if st != fa.FA_OK:
            raise fa.FaError(st, where)

    def step(ev):
        ev[0].record(stream)
        check(fa.fa_fwd(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                        scale, causal, sh), "fa_fwd")
        ev[1].record(stream)
        if w.backward:
            check(fa.fa_bwd_preprocess(o.data_ptr(), dog.data_ptr(), lse.data_ptr(), B, H, N, d, ws.data_ptr(),
                                       ws_bytes, sh), "fa_bwd_preprocess")
            ev[2].record(stream)
            check(fa.fa_bwd_dkdv(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), dog.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, N, d, scale, causal, ws.data_ptr(), ws_bytes, sh),
                  "fa_bwd_dkdv")
            ev[3].record(stream)
            check(fa.fa_bwd_dq_convert(dq.data_ptr(), B, H, N, d, scale, ws.data_ptr(), ws_bytes, sh),
                  "fa_bwd_dq_convert")
            ev[4].record(stream)

    launches_per_step = 4 if w.backward else 1
    nev = 5 if w.backward else 2
    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(nev)])
        if flush:
            flush_l2()
    torch.cuda.synchronize()
    check(fa.fa_get_device_status(sh), "warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    # Clock samples: nvidia-smi samples every 100 ms, longer than a short timed
    # region, so identical untimed steps keep the GPU busy for about half a
    # second before it and the samples cover that window plus the region.
    sampler = ClockSampler(local)
    sampler.start()
    spare = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    t_busy = time.perf_counter()
    busy_steps = 0
    while time.perf_counter() - t_busy < 0.6:
        step(spare)
        busy_steps += 1
        if busy_steps % 8 == 0:
            torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for i in range(args.steps):
        step(events[i])
        if flush and i + 1 < args.steps:
            flush_l2()   # outside the per-step events
    region1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = f"{busy_steps} untimed identical steps, then the timed region"
    check(fa.fa_get_device_status(sh), "timed region")

    step_ms = [e[0].elapsed_time(e[nev - 1]) for e in events]
    ms_per_step = sum(step_ms) / args.steps if flush else region0.elapsed_time(region1) / args.steps
    kern = {"fa_fwd_kernel": [e[0].elapsed_time(e[1]) for e in events]}
    if w.backward:
        kern["fa_bwd_pre"] = [e[1].elapsed_time(e[2]) for e in events]
        kern["fa_bwd_main"] = [e[2].elapsed_time(e[3]) for e in events]
        kern["fa_bwd_dq_conv"] = [e[3].elapsed_time(e[4]) for e in events]
    kern_avg = {k_: sum(v_) / len(v_) for k_, v_ in kern.items()}
    ms_per_step = max_over_ranks(ms_per_step, dev)
    fwd_f, bwd_f = flops_per_step(w)
    value = whole_job_tflops(world, fwd_f + bwd_f, ms_per_step)

    # ---- end to end: pinned host buffers in, results out, same C ABI ----
    # Every step copies its inputs in from pinned host memory and its results
    # out, as a serving or training loop would, pipelined over two device
    # buffer sets: step k+1's host-to-device copies (one stream) and step k-1's
    # device-to-host reads (another) overlap step k's kernels (a third).
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    n_sets = 2
    dev_in = [(qg, kg, vg, dog)] + [tuple(torch.empty_like(t) for t in (qg, kg, vg, dog)) for _ in range(n_sets - 1)]
    dev_out = [(o, lse, dq, dk, dv)] + [tuple(torch.empty_like(t) for t in (o, lse, dq, dk, dv))
                                        for _ in range(n_sets - 1)]
    host_out = [(torch.empty(q.shape, dtype=torch.bfloat16).pin_memory(),
                 torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
                 *(torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)))
                for _ in range(n_sets)]
    n_out = 5 if w.backward else 2
    h2d = sum(t.numel() * t.element_size() for t in ((hq, hk, hv, hdo) if w.backward else (hq, hk, hv)))
    d2h = sum(t.numel() * t.element_size() for t in host_out[0][:n_out])
    e2e_steps = max(2, min(args.steps, 10))
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cmp_h = s_cmp.cuda_stream

    def e2e_run(n):
        ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(n)]  # copied in, computed, copied out
        for i in range(n):
            st = i % n_sets
            qi, ki, vi, doi = dev_in[st]
            oi, lsei, dqi, dki, dvi = dev_out[st]
            with torch.cuda.stream(s_in):
                if i >= n_sets:
                    s_in.wait_event(ev[i - n_sets][1])  # the kernels of step i-2 are done with this set
                for hd, dd in ((hq, qi), (hk, ki), (hv, vi)) + (((hdo, doi),) if w.backward else ()):
                    dd.copy_(hd, non_blocking=True)
                ev[i][0].record(s_in)
            s_cmp.wait_event(ev[i][0])
            if i >= n_sets:
                s_cmp.wait_event(ev[i - n_sets][2])  # step i-2's results have left this set
            check(fa.fa_fwd(qi.data_ptr(), ki.data_ptr(), vi.data_ptr(), oi.data_ptr(), lsei.data_ptr(), B, H, N, d,
                            scale, causal, cmp_h), "fa_fwd")
            if w.backward:
                check(fa.fa_bwd(qi.data_ptr(), ki.data_ptr(), vi.data_ptr(), oi.data_ptr(), doi.data_ptr(),
                                lsei.data_ptr(), dqi.data_ptr(), dki.data_ptr(), dvi.data_ptr(), B, H, N, d, scale,
                                causal, ws.data_ptr(), ws_bytes, cmp_h), "fa_bwd")
            ev[i][1].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[i][1])
                for hd, dd in zip(host_out[st][:n_out], dev_out[st][:n_out]):
                    hd.copy_(dd, non_blocking=True)
                ev[i][2].record(s_out)

    e2e_run(n_sets)  # warm-up
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_run(e2e_steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = whole_job_tflops(world, fwd_f + bwd_f, e2e_ms)
    check(fa.fa_get_device_status(cmp_h), "e2e")

    # ---- the copies' own ceiling on this host: the same tensors moved with no
    # kernels, each direction alone and both at once (the e2e loop overlaps them)
    def copies(h2d_on, d2h_on, n):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        c0.record(s_in)
        s_out.wait_event(c0)
        for i in range(n):
            st = i % n_sets
            if h2d_on:
                with torch.cuda.stream(s_in):
                    for hd, dd in ((hq, dev_in[st][0]), (hk, dev_in[st][1]), (hv, dev_in[st][2])) + (
                            ((hdo, dev_in[st][3]),) if w.backward else ()):
                        dd.copy_(hd, non_blocking=True)
            if d2h_on:
                with torch.cuda.stream(s_out):
                    for hd, dd in zip(host_out[st][:n_out], dev_out[st][:n_out]):
                        hd.copy_(dd, non_blocking=True)
        s_in.wait_stream(s_out)
        c1.record(s_in)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / n
    copies(True, True, 1)
    # best of three rounds: the host side is shared, and a ceiling is the best the copies can do
    h2d_ms, d2h_ms, both_ms = (min(t) for t in zip(*[
        (copies(True, False, e2e_steps), copies(False, True, e2e_steps), copies(True, True, e2e_steps))
        for _ in range(3)]))
    e2e_ceiling = whole_job_tflops(world, fwd_f + bwd_f, max(ms_per_step, both_ms))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # ---- roofline of the dominant kernel ----
    peaks, peak_src = load_peaks()
    # Each pass against the measured dense bf16 peak (burst): the forward is its
    # one launch, the backward its three (preprocess, main, dQ convert).
    fwd_ms = kern_avg["fa_fwd_kernel"]
    bwd_ms = sum(kern_avg[k_] for k_ in ("fa_bwd_pre", "fa_bwd_main", "fa_bwd_dq_conv") if k_ in kern_avg)
    pass_fracs = {"fwd_ms": round(fwd_ms, 4), "fwd_tflops": round(fwd_f / (fwd_ms * 1e-3) / 1e12, 1),
                  "fwd_frac": round(fwd_f / (fwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    if w.backward:
        pass_fracs.update({"bwd_ms": round(bwd_ms, 4), "bwd_tflops": round(bwd_f / (bwd_ms * 1e-3) / 1e12, 1),
                           "bwd_frac": round(bwd_f / (bwd_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)})
    pass_fracs["frac_peak"] = f"{peaks['bf16_tflops']} TFLOP/s, {peak_src} dense bf16 (burst)"
    dom = max(kern_avg, key=kern_avg.get)
    per_launch = {"fa_fwd_kernel": fwd_f, "fa_bwd_main": bwd_f}
    if dom in per_launch:
        achieved = per_launch[dom] / (kern_avg[dom] * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4)}
    else:
        bytes_ = (2 * w.B * w.H * w.N * w.d * 2 + 8 * w.B * w.H * w.N if dom == "fa_bwd_pre"
                  else w.B * w.H * w.N * w.d * 6)
        achieved = bytes_ / (kern_avg[dom] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
    roof["traffic"] = dram_traffic(dom, w.name)
    roof["peak_source"] = f"{peak_src} (burst bf16 GEMM)" if roof["bound"] == "tensor" else peak_src
    roof["kernel_ms"] = {k_: round(v_, 4) for k_, v_ in kern_avg.items()}
    roof["kernel_frac_of_peak"] = {
        k_: round(per_launch[k_] / (kern_avg[k_] * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
        for k_ in kern_avg if k_ in per_launch}

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**w.describe(), "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": ("flushed between steps (2x L2 buffer written, then another read)" if flush
                              else "inputs larger than L2 (each tensor > 129 MB)"),
                       "fwd_tflop_per_step": round(fwd_f / 1e12, 4), "bwd_tflop_per_step": round(bwd_f / 1e12, 4),
                       **pass_fracs,
                       "pct_of_dense_bf16_2250": round(100 * value / world / 2250.0, 2),
                       "pct_of_measured_bf16": round(100 * value / world / peaks["bf16_tflops"], 2)},
            "roofline": roof, "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
            "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "pipelining": "2 device buffer sets; step k+1's host-to-device and step k-1's "
                                  "device-to-host copies overlap step k's kernels",
                    "copy_gbs_ceiling": {"h2d_alone": round(h2d / (h2d_ms * 1e-3) / 1e9, 1),
                                         "d2h_alone": round(d2h / (d2h_ms * 1e-3) / 1e9, 1),
                                         "both_at_once_ms_per_step": round(both_ms, 4)},
                    "ceiling": round(e2e_ceiling, 3),
                    "ceiling_is": "the metric at max(device step, both directions' copies at once)",
                    "frac_of_ceiling": round(e2e_value / e2e_ceiling, 4)}}
    if world == 1 and not args.no_cpu_baseline:
        val, n, el = oracle_sample(w, q, k, v, do, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(val, 6), "unit": UNIT, "cores": cores(), "kind": "oracle",
                                "sample": f"{n} unit(s) of up to {ORACLE_ROWS} query rows of one (b,h) slice "
                                          f"(fwd{' + its share of the bwd' if w.backward else ''}) of "
                                          f"{len(oracle_units(w))} in the workload, fp64 numpy, {el:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


DECODE_METRIC = "split-KV decode forward: K/V cache read GB/s (1 GPU)"


def decode_bytes(w):
    """Algorithmic HBM bytes of one decode step: read Q, K, V; write O and lse."""
    return 2 * w.B * w.H * w.Nk * w.d * 2 + 2 * w.B * w.H * w.Nq * w.d * 2 + 4 * w.B * w.H * w.Nq


def run_decode(args, w):
    """Split-KV decode forward (fa_fwd_splitkv): device-timed GB/s against the HBM roofline."""
    import exact_io_aware_31_gb300 as fa
    from exact_io_aware_31_gb300 import build

    rank, world, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    build.build()
    fa.load_library()
    q, k, v = workloads.make_decode_inputs(w.B, w.H, w.Nq, w.Nk, w.d, w.seed)
    dev = torch.device("cuda", local)
    qg, kg, vg = (t.to(dev) for t in (q, k, v))
    o = torch.empty_like(qg)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    splits = 0
    ws_bytes = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, splits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    flush_l2 = L2Flush(dev)

    def step():
        st = fa.fa_fwd_splitkv(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H,
                               w.Nq, w.Nk, w.d, w.scale, int(w.causal), splits, ws.data_ptr(), ws_bytes, sh)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_splitkv")

    for _ in range(args.warmup):
        step()
        flush_l2()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_busy = time.perf_counter()
    busy = 0
    while time.perf_counter() - t_busy < 0.6:
        step()
        busy += 1
        if busy % 32 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in events:
        flush_l2()   # the cache is about L2-sized: every timed step reads it from HBM
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = f"{busy} untimed identical steps, then the timed region"
    if fa.fa_get_device_status(sh) != fa.FA_OK:
        raise RuntimeError("device status after the timed region")
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in events)
    nbytes = decode_bytes(w)
    value = nbytes / (ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    # ---- end to end: the cache and queries from pinned host memory, results back ----
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32).pin_memory()

    def e2e_step():
        for hd, dd in ((hq, qg), (hk, kg), (hv, vg)):
            dd.copy_(hd, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 10))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * 2 + hlse.numel() * 4
    launches = 1 if ws_bytes == 0 else 2
    line = {"metric": DECODE_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate", "data": "synthetic",
            "config": {**w.describe(), "parallelism": "single GPU",
                       "splits": "chosen by the library (num_splits = 0)",
                       "merge": ("no workspace (one split per head, or a head's splits merge in one cluster)"
                                 if ws_bytes == 0 else "workspace + merge kernel"),
                       "l2": "flushed before every timed step (2x L2 buffer written, then another read)",
                       "bytes_per_step": nbytes},
            "roofline": {"kernel": "fa_decode_split (+ fa_decode_combine)", "bound": "hbm",
                         "achieved": round(value, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(value / peaks["hbm_gbs"], 4), "traffic": None, "peak_source": peak_src},
            "gpu_launches": launches * args.steps, "clocks": clocks,
            "e2e": {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps}}
    if not args.no_cpu_baseline:
        import numpy as np
        from oracle.decode import attention_forward_rect
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < args.cpu_seconds and n < w.B * w.H:
            b, h = divmod(n, w.H)
            attention_forward_rect(*(t[b:b + 1, h:h + 1].double().numpy() for t in (q, k, v)), w.scale, w.causal)
            n += 1
        el = time.perf_counter() - t0
        cpu_gbs = nbytes * n / (w.B * w.H) / el / 1e9
        line["cpu_baseline"] = {"value": round(cpu_gbs, 4), "unit": "GB/s", "cores": cores(), "kind": "oracle",
                                "sample": f"{n} of {w.B * w.H} heads in fp64 numpy, {el:.1f} s"}
    print(json.dumps(line), flush=True)


FP8_METRIC = "attention forward with E4M3 Q, K: TFLOP/s (1 GPU)"


def run_fp8(args, w):
    """Forward with E4M3 queries and keys (fa_fwd_fp8), device-timed, d = 128 workloads.

    Half of the forward's FLOPs (S = Q K^T) run in E4M3, half (P V) in bf16;
    at the nominal 2:1 ratio of the E4M3 and bf16 dense rates the mix's peak
    is 4/3 of the measured bf16 peak, the denominator reported here.
    """
    import exact_io_aware_31_gb300 as fa
    from exact_io_aware_31_gb300 import build

    rank, world, local = dist_env()
    if rank != 0:
        return
    if w.d != 128:
        raise SystemExit("--fp8 needs a d = 128 workload")
    torch.cuda.set_device(local)
    build.build()
    fa.load_library()
    q8, k8, qs, ks, v = workloads.make_fp8_inputs(w.B, w.H, w.N, w.d, w.seed)
    dev = torch.device("cuda", local)
    qg, kg, vg = (t.to(dev) for t in (q8, k8, v))
    o = torch.empty_like(vg)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    flush_l2 = L2Flush(dev)

    def step():
        st = fa.fa_fwd_fp8(qg.data_ptr(), kg.data_ptr(), vg.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N,
                           w.d, w.scale, qs, ks, int(w.causal), sh)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd_fp8")

    for _ in range(args.warmup):
        step()
        flush_l2()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in events:
        flush_l2()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if fa.fa_get_device_status(sh) != fa.FA_OK:
        raise RuntimeError("device status after the timed region")
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in events)
    fwd, _ = flops_per_step(w)
    tflops = fwd / (ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"] * 4.0 / 3.0
    hq, hk, hv = (t.pin_memory() for t in (q8, k8, v))
    ho = torch.empty(v.shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()

    def e2e_step():
        for hd, dd in ((hq, qg), (hk, kg), (hv, vg)):
            dd.copy_(hd, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 10))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a0.elapsed_time(a1) / e2e_steps
    line = {"metric": FP8_METRIC, "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 Q K, bf16 V P O, fp32 accumulate", "data": "synthetic",
            "config": {**w.describe(), "backward": False, "parallelism": "single GPU",
                       "inputs": "Q, K per-tensor scaled E4M3 codes (descale = max|x| / 448)",
                       "l2": "flushed before every timed step (2x L2 buffer written, then another read)"},
            "roofline": {"kernel": "fa_fwd_kernel (E4M3 S)", "bound": "tensor", "achieved": round(tflops, 1),
                         "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": dram_traffic("fa_fwd_kernel_fp8", w.name),
                         "peak_source": peak_src + " bf16 x 4/3 (half the FLOPs at 2x rate)"},
            "gpu_launches": args.steps, "clocks": clocks,
            "e2e": {"value": round(fwd / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hk, hv)),
                    "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4, "steps": e2e_steps}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.LONG_SEQ.name,
                    help="one of: " + ", ".join(sorted(workloads.BY_NAME) + sorted(workloads.DECODE_BY_NAME)))
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true", help="forward with E4M3 Q, K (fa_fwd_fp8) on a d = 128 workload")
    args = ap.parse_args()
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.workload in workloads.DECODE_BY_NAME:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the forward/backward "
                              "workloads; the decode row reports its oracle under cpu_baseline"}))
            return
        run_decode(args, workloads.DECODE_BY_NAME[args.workload])
        return
    w = workloads.BY_NAME[args.workload]
    if args.fp8:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the bf16 "
                              "forward/backward workloads"}))
            return
        run_fp8(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
