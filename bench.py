#!/usr/bin/env python3
"""Benchmark of the causal depthwise conv1d forward pass on GB300.

One step = one forward pass over the whole workload (one kernel launch).  The
default workload is the bf16 Mamba-style prefill, B=8, C=5120, L=2048, K=4,
SiLU, contiguous [B,C,L].  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5|all]
                  [--impl ours|reference] [--op fwd|update|bwd]

``--op update`` times the decode step and ``--op bwd`` the backward pass
(gradient kernel + partial-sum reduction) on the same workloads; the default
(``fwd``) is the contract line described here.

``value``: algorithmic bytes (x read + out written + weight + bias + states +
seq_idx, each once) per second over the timed region, inputs resident in HBM.
Consecutive steps rotate over four buffer sets, so every step streams its
input from HBM (each set is larger than the 129 MB L2 cache).
``roofline.achieved``: the same bytes per launch divided by the mean launch
duration, the timed region's CUDA-event time over its launches (one launch
per step, issued back to back with events only at the region's ends;
``kernel_bracketed_us`` gives the mean of launches each between two events of
its own, which serialises them, for context).
``e2e``: the same metric through the public API with host buffers, the
host-to-device copy of x and the device-to-host copy of out inside the timed
region.
``per_config`` (default run, rank 0; ``--no-per-config`` leaves it out): each
of the five workloads timed the same way over 2000 back-to-back launches with
its own clock samples, every output of its last launch compared with the
oracle, and ``layout_copy``: the framework's own ``copy_`` of the same input
view into the same output buffer (x read + out written, no arithmetic),
timed the same way, as a reference for what the memory system gives that
layout.
``--impl reference``: the CPU oracle (the plain single-threaded FP64
implementation the tests compare against), timed on this host's cores on a
bounded sample of the same workload.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the operation has no cross-GPU exchange); ``value`` counts the
bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal_conv1d_fwd HBM GB/s (in+out bytes) and % of GB300 HBM roofline"
FALLBACK_HBM_GBS = 6800.0
N_SETS = 4

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture,
# keyed by a hash of the kernel sources it was taken on (stale -> null).
NCU_TRAFFIC = {
    "20c53cc462e38675": {
        "c2_bf16_contig_B8_C5120_L2048_K4_silu": 291081728,
        "c3_bf16_chlast_view_B4_C5120_L4096_K4_silu_states": 287014144,
        "c4_f16_chlast_B1_C4096_L16384_K4_silu_seqidx": 218449920,
        "c5_f32_contig_B1_C16_L4194304_K3_final": 483036160,
        "c2_bf16_contig_B8_C5120_L2048_K4_silu_bwd": 465957120,
        "c3_bf16_chlast_view_B4_C5120_L4096_K4_silu_states_bwd": 482709504,
        "c4_f16_chlast_B1_C4096_L16384_K4_silu_seqidx_bwd": 379876352,
        "c5_f32_contig_B1_C16_L4194304_K3_final_bwd": 763793664,
    },
}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "causal_depthwise_conv1d_gb300", "csrc", "*"))):
        with open(p, "rb") as fh:
            h.update(os.path.basename(p).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy_ of 1 Gi bf16, burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def nominal_hbm_gbs(local: int):
    """2 x memory clock x bus width / 8 from the CUDA runtime's device
    attributes (memory clock in kHz, bus width in bits), or None when the
    runtime does not report them."""
    import ctypes
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for name in ("libcudart.so", os.path.join(cuda_home, "lib64", "libcudart.so"), "libcudart.so.13"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    else:
        return None
    clock_khz, bus_bits = ctypes.c_int(0), ctypes.c_int(0)
    if rt.cudaDeviceGetAttribute(ctypes.byref(clock_khz), 36, local) != 0:  # cudaDevAttrMemoryClockRate
        return None
    if rt.cudaDeviceGetAttribute(ctypes.byref(bus_bits), 37, local) != 0:  # cudaDevAttrGlobalMemoryBusWidth
        return None
    if clock_khz.value <= 0 or bus_bits.value <= 0:
        return None
    return 2.0 * clock_khz.value * 1e3 * bus_bits.value / 8 / 1e9


def smi_index(local: int) -> str:
    """nvidia-smi index of this process's CUDA device `local` (the entry of
    CUDA_VISIBLE_DEVICES when it is set)."""
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    return vis[local] if local < len(vis) else str(local)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world):
    """Max over ranks of a list of floats (identity for one rank)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def measure_copy_bw(torch, device) -> float:
    """D2D copy bandwidth (read + write bytes) of a 1 Gi-element bf16 copy, best of 10."""
    n = 1 << 30
    a = torch.empty(n, dtype=torch.bfloat16, device=device)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = float("inf")
    for _ in range(3):
        b.copy_(a)
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        b.copy_(a)
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e) / 1e3)
    del a, b
    torch.cuda.empty_cache()
    return 2 * n * 2 / best / 1e9


def prepare_sets(torch, p, device, n_sets):
    """n_sets independent device copies of the workload, pre-marshalled for the C ABI."""
    import ctypes
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding, device as dv

    lib = ccv.load_library()
    base = dv.to_device(p, device=device)
    stream = torch.cuda.current_stream(device)
    sets = []
    for i in range(n_sets):
        d = base if i == 0 else dv.to_device(p, device=device)
        arr = binding._arr
        args = (ctypes.c_void_p(d.x.data_ptr()), arr(d.x.stride()),
                ctypes.c_void_p(d.out.data_ptr()), arr(d.out.stride()),
                ctypes.c_void_p(d.weight.data_ptr()), arr(d.weight.stride()),
                ctypes.c_void_p(d.bias.data_ptr()) if d.bias is not None else None,
                ctypes.c_int64(d.bias.stride(0) if d.bias is not None else 0),
                ctypes.c_void_p(d.seq_idx.data_ptr()) if d.seq_idx is not None else None,
                arr(d.seq_idx.stride()) if d.seq_idx is not None else None,
                ctypes.c_void_p(d.initial_states.data_ptr()) if d.initial_states is not None else None,
                arr(d.initial_states.stride()) if d.initial_states is not None else None,
                ctypes.c_void_p(d.final_states.data_ptr()) if d.final_states is not None else None,
                arr(d.final_states.stride()) if d.final_states is not None else None,
                ctypes.c_int64(p.B), ctypes.c_int64(p.C), ctypes.c_int64(p.L), ctypes.c_int(p.K),
                ctypes.c_int(binding.TORCH_DTYPE[d.x.dtype]),
                ctypes.c_int(1 if p.activation_silu else 0), ctypes.c_void_p(stream.cuda_stream))
        sets.append((d, args))
    return lib, sets


TIMING_NOTE = ("timed region: back-to-back launches on one stream with an event at each end; each kernel is "
               "launched with programmatic stream serialization, so its launch and block ramp-up overlap the "
               "previous launch's tail; *_bracketed_us: the same launches each between two events of its own, "
               "which serialises them (context)")


def bracketed_mean(torch, stream, launch, steps, most=200):
    """Mean time of up to `most` launches, each recorded between two events
    of its own (outside the timed region; context for the region's mean)."""
    n = max(1, min(steps, most))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        ev[i][0].record(stream)
        launch(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / 1e3 / n


def measure_e2e(torch, ccv, p, sets, stream, args, world, nbytes):
    """Public API with host buffers, as a streaming user runs it: every step
    copies its x from pinned host memory, runs ccv_fwd and copies its out back
    to pinned host memory.  Consecutive steps are pipelined on three streams
    (copy in, compute, copy out) over two device buffer sets and two host
    output buffers, with events ordering each step's copy-in, kernel and
    copy-out and the reuse of a set two steps later."""
    d_sets = [sets[0][0], sets[1 % len(sets)][0]]
    x_host = d_sets[0].x_buf.cpu().pin_memory()
    w_host = d_sets[0].weight.cpu().pin_memory()
    b_host = d_sets[0].bias.cpu().pin_memory() if d_sets[0].bias is not None else None
    out_host = [torch.empty(d.out_buf.shape, dtype=d.out_buf.dtype).pin_memory() for d in d_sets]
    e2e_steps = max(4, min(args.steps, 50))
    h2d = x_host.numel() * x_host.element_size() + w_host.numel() * w_host.element_size() + (
        b_host.numel() * b_host.element_size() if b_host is not None else 0)
    d2h = out_host[0].numel() * out_host[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    k_done = [None, None]
    o_done = [None, None]

    def step(i):
        j = i % 2
        d = d_sets[j]
        with torch.cuda.stream(s_in):
            if k_done[j] is not None:
                s_in.wait_event(k_done[j])  # the kernel two steps back has read this set's x
            d.x_buf.copy_(x_host, non_blocking=True)
            d.weight.copy_(w_host, non_blocking=True)
            if b_host is not None:
                d.bias.copy_(b_host, non_blocking=True)
            in_done = ev()
            in_done.record(s_in)
        stream.wait_event(in_done)
        if o_done[j] is not None:
            stream.wait_event(o_done[j])  # the copy-out two steps back has read this set's out
        ccv.ccv_fwd(d.x, d.weight, d.bias, d.seq_idx, d.initial_states, final_states_out=d.final_states,
                    activation=p.activation, out=d.out, stream=stream)
        k_done[j] = ev()
        k_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(k_done[j])
            out_host[j].copy_(d.out_buf, non_blocking=True)
            o_done[j] = ev()
            o_done[j].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    k_done[:] = [None, None]
    o_done[:] = [None, None]
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(s_in)
    for i in range(e2e_steps):
        step(i)
    s_out.wait_event(k_done[(e2e_steps - 1) % 2])
    ee.record(s_out)
    torch.cuda.synchronize()
    e2e_s = es.elapsed_time(ee) / 1e3 / e2e_steps

    # Ceiling of the host link: the same two copies with no kernel, both
    # directions at once (what the pipelined steady state needs).
    def copies():
        with torch.cuda.stream(s_in):
            d_sets[1].x_buf.copy_(x_host, non_blocking=True)
        with torch.cuda.stream(s_out):
            out_host[1].copy_(d_sets[0].out_buf, non_blocking=True)

    copies()
    torch.cuda.synchronize()
    reps = 5
    cs, ce = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cs.record(s_in)
    s_out.wait_event(cs)
    for _ in range(reps):
        copies()
    out_fin = ev()
    out_fin.record(s_out)
    s_in.wait_event(out_fin)
    ce.record(s_in)
    torch.cuda.synchronize()
    link_s = cs.elapsed_time(ce) / 1e3 / reps
    (e2e_s, link_s) = reduce_max([e2e_s, link_s], world)
    per_dir = max(h2d, d2h)
    return {"value": round(world * nbytes / e2e_s / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "pipelined": "copy-in, kernel and copy-out of consecutive steps overlap (3 streams, 2 buffer sets)",
            "host_link": {"e2e_GBps_each_way": round(per_dir / e2e_s / 1e9, 1),
                          "concurrent_copy_GBps_each_way": round(per_dir / link_s / 1e9, 1),
                          "frac": round(link_s / e2e_s, 3),
                          "note": "the step's H2D and D2H copies alone, both directions at once, pinned buffers"}}


def run_ours(args, p, world, rank, local):
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    ccv.load_library()
    hbm_peak, peak_source = load_peaks()
    copy_bw = None if args.skip_extras else measure_copy_bw(torch, device)
    nominal = nominal_hbm_gbs(local)
    n_sets = max(1, args.sets)
    lib, sets = prepare_sets(torch, p, device, n_sets)
    nbytes = p.algorithmic_bytes()

    def launch(i):
        rc = lib.ccv_fwd(*sets[i % n_sets][1])
        if rc != 0:
            raise RuntimeError(ccv.ccv_last_error())

    for i in range(args.warmup):
        launch(i)
    kernel_name = ccv.ccv_last_kernel()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(smi_index(local))
    sampler.start()
    time.sleep(0.2)
    stream = torch.cuda.current_stream(device)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_begin.record(stream)
    for i in range(args.steps):
        launch(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_s = t_begin.elapsed_time(t_end) / 1e3
    # one launch per step, back to back: the mean launch duration is the
    # region's time over its launches
    mean_launch = total_s / args.steps
    bracketed = bracketed_mean(torch, stream, launch, args.steps)
    total_s, mean_launch, bracketed = reduce_max([total_s, mean_launch, bracketed], world)

    e2e = None
    if not args.skip_extras:
        e2e = measure_e2e(torch, ccv, p, sets, stream, args, world, nbytes)
    result = {
        "metric": METRIC,
        "value": round(world * nbytes * args.steps / total_s / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_s / args.steps * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": p.name, "io_dtype": p.dtype, "B": p.B, "C": p.C, "L": p.L, "K": p.K,
                   "activation": p.activation or "none", "x_strides": list(p.x_strides),
                   "seq_idx": p.seq_idx is not None, "initial_states": p.init_buf is not None,
                   "final_states": p.want_final, "algorithmic_bytes_per_step": nbytes,
                   "l2": f"inputs larger than L2; {n_sets} rotating buffer sets",
                   "parallelism": "replica per GPU" if world > 1 else "single GPU",
                   "kernel": kernel_name, "recipe": p.recipe},
        "gelem_per_s": round(world * p.B * p.C * p.L * args.steps / total_s / 1e9, 3),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / mean_launch / 1e9, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(nbytes / mean_launch / 1e9 / hbm_peak, 4),
                     "traffic": NCU_TRAFFIC.get(kernel_source_hash(), {}).get(p.name),
                     "peak_source": peak_source, "kernel_mean_us": round(mean_launch * 1e6, 3),
                     "kernel_bracketed_us": round(bracketed * 1e6, 3), "timing": TIMING_NOTE},
        "nominal_hbm": None if nominal is None else {
            "value": round(nominal, 1), "unit": "GB/s", "frac": round(nbytes / mean_launch / 1e9 / nominal, 4),
            "source": "2 x memory clock x bus width / 8, CUDA device attributes"},
        "copy_bw_same_run": None if copy_bw is None else {
            "value": round(copy_bw, 1), "unit": "GB/s", "frac": round(nbytes / mean_launch / 1e9 / copy_bw, 4)},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    out_dev = sets[(args.steps - 1) % n_sets][0]
    return result, out_dev


def cpu_baseline_and_parity(p, out_dev, budget_s=20.0):
    """Time the oracle single-threaded on a bounded sample (whole rows) and
    compare the GPU output on that sample."""
    import numpy as np
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import compare
    from oracle import oracle as orc

    rows_total = p.B * p.C
    # calibrate on one batch row block
    probe_c = max(1, min(p.C, 64))
    x = p.x_view()
    init = p.init_view()
    t0 = time.perf_counter()
    orc.causal_conv1d_fwd(x[:1, :probe_c], p.weight[:probe_c], None if p.bias is None else p.bias[:probe_c],
                          p.dtype, p.activation, None if p.seq_idx is None else p.seq_idx[:1],
                          None if init is None else init[:1, :probe_c], p.want_final)
    per_row = (time.perf_counter() - t0) / probe_c
    rows = int(max(1, min(rows_total, budget_s / max(per_row, 1e-9))))
    nb = max(1, min(p.B, rows // p.C)) if rows >= p.C else 1
    nc = p.C if rows >= p.C else rows
    t0 = time.perf_counter()
    ref, ref_fin, _ = orc.causal_conv1d_fwd(
        x[:nb, :nc], p.weight[:nc], None if p.bias is None else p.bias[:nc], p.dtype, p.activation,
        None if p.seq_idx is None else p.seq_idx[:nb], None if init is None else init[:nb, :nc], p.want_final)
    secs = time.perf_counter() - t0
    e = {"f32": 4, "f16": 2, "bf16": 2}[p.dtype]
    sample_bytes = 2 * nb * nc * p.L * e
    got = dv.torch_to_host(out_dev.out[:nb, :nc], p.dtype)
    rep = compare.compare_out(got, ref, p.dtype)
    fin_ok = None
    if p.want_final and out_dev.final_states is not None:
        fin_ok = compare.compare_bits(dv.torch_to_host(out_dev.final_states[:nb, :nc], p.dtype), ref_fin) == 0
    base = {"value": round(sample_bytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"x[:{nb}, :{nc}, :] of the workload ({nb * nc} of {rows_total} rows, "
                      f"{nb * nc * p.L} outputs), {secs:.1f} s, single-threaded C oracle (FP64)",
            "host_cores_available": os.cpu_count(), "host_cpu": host_cpu_model()}
    par = {"outputs_checked": rep.n, "outside_tolerance": rep.n_bad, "max_err": rep.max_err,
           "max_err_unit": "abs" if p.dtype == "f32" else "ulp", "final_states_bit_exact": fin_ok}
    del np
    return base, par


def host_cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm
    implementer and part codes), else the machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as fh:
            info = fh.read()
    except OSError:
        return platform.machine()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.machine()


def oracle_threads(p, threads=0):
    """The oracle over the whole workload, channel ranges in parallel threads
    (each range an ordinary single-threaded oracle call; the C oracle releases
    the GIL)."""
    import concurrent.futures as cf
    import numpy as np
    from oracle import oracle as orc

    threads = threads or min(32, os.cpu_count() or 1)
    x = p.x_view()
    init = p.init_view()
    bounds = np.linspace(0, p.C, min(threads, p.C) + 1).astype(int)

    def run(lo, hi):
        o, f, _ = orc.causal_conv1d_fwd(
            x[:, lo:hi, :], p.weight[lo:hi], None if p.bias is None else p.bias[lo:hi], p.dtype, p.activation,
            p.seq_idx, None if init is None else init[:, lo:hi, :], p.want_final, weight_dtype=p.wdt)
        return o, f

    with cf.ThreadPoolExecutor(max_workers=len(bounds) - 1) as ex:
        parts = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    out = np.concatenate([o for o, _ in parts], axis=1)
    fin = np.concatenate([f for _, f in parts], axis=1) if p.want_final else None
    return out, fin


def per_config_record(local, launches=2000):
    """Every workload on this GPU: `launches` back-to-back launches (the same
    timing as the headline: events at the region's two ends, four rotating
    buffer sets larger than L2, clocks sampled during the region) and every
    output of the last launch compared with the oracle."""
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from causal_depthwise_conv1d_gb300 import inputs
    from oracle import compare

    device = torch.device("cuda", local)
    peak, _ = load_peaks()
    rec = {}
    for idx in (1, 2, 3, 4, 5):
        p = inputs.make_config(idx)
        lib, sets = prepare_sets(torch, p, device, N_SETS)
        nbytes = p.algorithmic_bytes()

        def launch(i):
            rc = lib.ccv_fwd(*sets[i % N_SETS][1])
            if rc != 0:
                raise RuntimeError(ccv.ccv_last_error())

        for i in range(20):
            launch(i)
        kernel = ccv.ccv_last_kernel()
        torch.cuda.synchronize()
        sampler = ClockSampler(smi_index(local))
        sampler.start()
        time.sleep(0.2)
        stream = torch.cuda.current_stream(device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(launches):
            launch(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        clocks = sampler.stop()
        mean = ev0.elapsed_time(ev1) / 1e3 / launches
        out_dev = sets[(launches - 1) % N_SETS][0]
        got = dv.torch_to_host(out_dev.out, p.dtype)
        ref, ref_fin = oracle_threads(p)
        rep = compare.compare_out(got, ref, p.dtype)
        fin_ok = None
        if p.want_final and out_dev.final_states is not None:
            fin_ok = compare.compare_bits(dv.torch_to_host(out_dev.final_states, p.dtype), ref_fin) == 0
        # reference: the framework's own copy of the same input view into the
        # same output buffer (x read + out written, no arithmetic), timed the
        # same way
        copy_launches = 300
        for i in range(10):
            sets[i % N_SETS][0].out.copy_(sets[i % N_SETS][0].x)
        ev0.record(stream)
        for i in range(copy_launches):
            sets[i % N_SETS][0].out.copy_(sets[i % N_SETS][0].x)
        ev1.record(stream)
        torch.cuda.synchronize()
        copy_us = ev0.elapsed_time(ev1) * 1e3 / copy_launches
        copy_bytes = 2 * p.B * p.C * p.L * (4 if p.dtype == "f32" else 2)
        gbs = nbytes / mean / 1e9
        rec[p.name] = {"kernel": kernel, "launches": launches, "kernel_mean_us": round(mean * 1e6, 3),
                       "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                       "gelem_per_s": round(p.B * p.C * p.L / mean / 1e9, 2),
                       "algorithmic_bytes": nbytes,
                       "parity": {"outputs_checked": rep.n, "outside_tolerance": rep.n_bad,
                                  "max_err": rep.max_err, "max_err_unit": "abs" if p.dtype == "f32" else "ulp",
                                  "final_states_bit_exact": fin_ok},
                       "clocks": clocks,
                       "layout_copy": {"us": round(copy_us, 3), "frac": round(copy_bytes / copy_us / 1e3 / peak, 4),
                                       "what": "torch copy_ of the same input view into the same output buffer"}}
        del sets, out_dev, got, ref
        torch.cuda.empty_cache()
    return rec


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args, p):
    from oracle import oracle as orc

    orc.build()
    x = p.x_view()
    init = p.init_view()
    e = {"f32": 4, "f16": 2, "bf16": 2}[p.dtype]
    # rows per step: the whole --warmup + --steps run stays within ~120 s
    t0 = time.perf_counter()
    probe_c = max(1, min(p.C, 16))
    orc.causal_conv1d_fwd(x[:1, :probe_c], p.weight[:probe_c], None if p.bias is None else p.bias[:probe_c],
                          p.dtype, p.activation, None if p.seq_idx is None else p.seq_idx[:1],
                          None if init is None else init[:1, :probe_c], p.want_final)
    per_row = (time.perf_counter() - t0) / probe_c
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(p.C, budget / max(per_row, 1e-9))))

    def step(i):
        c0 = (i * rows) % p.C
        c1 = min(p.C, c0 + rows)
        b = (i * rows // p.C) % p.B
        orc.causal_conv1d_fwd(x[b:b + 1, c0:c1], p.weight[c0:c1], None if p.bias is None else p.bias[c0:c1],
                              p.dtype, p.activation, None if p.seq_idx is None else p.seq_idx[b:b + 1],
                              None if init is None else init[b:b + 1, c0:c1], p.want_final)
        return (c1 - c0) * p.L

    for i in range(args.warmup):
        step(i)
    n = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        n += step(args.warmup + i)
    secs = time.perf_counter() - t0
    value = 2 * n * e / secs / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": p.name, "io_dtype": p.dtype, "B": p.B, "C": p.C, "L": p.L, "K": p.K,
                   "activation": p.activation or "none"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle", "cores": 1,
                         "sample": f"each step: {rows} channel rows x {p.L} steps of the workload",
                         "host_cores_available": os.cpu_count(), "host_cpu": host_cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def bwd_algorithmic_bytes(p) -> int:
    """x and dout read, dx written, weight / bias read and their gradients
    written, states and dfinal_states / dinitial_states, seq_idx: each once."""
    e = {"f32": 4, "f16": 2, "bf16": 2}[p.dtype]
    n = p.B * p.C * p.L
    total = 3 * n * e + 2 * p.C * p.K * e
    if p.bias is not None:
        total += 2 * p.C * e
    if p.seq_idx is not None:
        total += p.B * p.L * 4
    if p.init_buf is not None:
        total += 2 * p.B * p.C * (p.K - 1) * e
    if p.want_final:
        total += p.B * p.C * (p.K - 1) * e
    return total


def run_bwd_bench(args, p, world, local):
    """Backward pass (ccv_bwd: gradient kernel + partial-sum reduction) on a
    workload: dout ~ N(0,1) in x's layout, dfinal_states when the forward
    returns final states, every gradient requested."""
    import ctypes
    import numpy as np
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding, inputs
    from causal_depthwise_conv1d_gb300 import device as dv

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    lib = ccv.load_library()
    hbm_peak, peak_source = load_peaks()
    rng = np.random.default_rng(1)
    g_np = inputs.round_to_storage(rng.standard_normal(p.x_buf.size), p.dtype)
    g_host = dv.host_to_torch(g_np, p.dtype)
    dfin_np = dfin_host = None
    if p.want_final:
        dfin_np = inputs.round_to_storage(rng.standard_normal((p.B, p.C, p.K - 1)), p.dtype)
        dfin_host = dv.host_to_torch(dfin_np, p.dtype)
    stream = torch.cuda.current_stream(device)
    arr = binding._arr
    n_sets = 2
    sets = []
    for _ in range(n_sets):
        d = dv.to_device(p, device=device)
        gbuf = g_host.to(device)
        dout = gbuf.as_strided((p.B, p.C, p.L), p.x_strides, p.x_offset)
        dfin = dfin_host.to(device) if dfin_host is not None else None
        dx = binding._dense_like_fast_dim(d.x, p.B, p.C, p.L)
        dw = torch.empty((p.C, p.K), dtype=d.x.dtype, device=device)
        db = torch.empty((p.C,), dtype=d.x.dtype, device=device) if p.bias is not None else None
        di = torch.empty((p.B, p.C, p.K - 1), dtype=d.x.dtype, device=device) if p.init_buf is not None else None
        need = ccv.ccv_bwd_workspace_size(d.x.stride(), dout.stride(), dx.stride(), p.B, p.C, p.L, p.K,
                                          binding.TORCH_DTYPE[d.x.dtype])
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=device)
        keep = (d, gbuf, dfin, dx, dw, db, di, ws)
        call = (ctypes.c_void_p(d.x.data_ptr()), arr(d.x.stride()), ctypes.c_void_p(d.weight.data_ptr()),
                arr(d.weight.stride()), ctypes.c_void_p(d.bias.data_ptr()) if d.bias is not None else None,
                ctypes.c_int64(1), ctypes.c_void_p(d.seq_idx.data_ptr()) if d.seq_idx is not None else None,
                arr(d.seq_idx.stride()) if d.seq_idx is not None else None,
                ctypes.c_void_p(d.initial_states.data_ptr()) if d.initial_states is not None else None,
                arr(d.initial_states.stride()) if d.initial_states is not None else None,
                ctypes.c_void_p(dout.data_ptr()), arr(dout.stride()),
                ctypes.c_void_p(dfin.data_ptr()) if dfin is not None else None,
                arr(dfin.stride()) if dfin is not None else None,
                ctypes.c_void_p(dx.data_ptr()), arr(dx.stride()), ctypes.c_void_p(dw.data_ptr()), arr(dw.stride()),
                ctypes.c_void_p(db.data_ptr()) if db is not None else None, ctypes.c_int64(1),
                ctypes.c_void_p(di.data_ptr()) if di is not None else None,
                arr(di.stride()) if di is not None else None, ctypes.c_void_p(ws.data_ptr()),
                ctypes.c_uint64(ws.numel()), ctypes.c_int64(p.B), ctypes.c_int64(p.C), ctypes.c_int64(p.L),
                ctypes.c_int(p.K), ctypes.c_int(binding.TORCH_DTYPE[d.x.dtype]),
                ctypes.c_int(1 if p.activation_silu else 0), ctypes.c_void_p(stream.cuda_stream))
        sets.append((keep, call, need))

    def launch(i):
        rc = lib.ccv_bwd(*sets[i % n_sets][1])
        if rc != 0:
            raise RuntimeError(ccv.ccv_last_error())

    for i in range(args.warmup):
        launch(i)
    kernel_name = ccv.ccv_last_kernel()
    torch.cuda.synchronize()
    sampler = ClockSampler(smi_index(local))
    sampler.start()
    time.sleep(0.2)
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_begin.record(stream)
    for i in range(args.steps):
        launch(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    total_s = t_begin.elapsed_time(t_end) / 1e3
    mean_step = total_s / args.steps
    bracketed = bracketed_mean(torch, stream, launch, args.steps)
    nbytes = bwd_algorithmic_bytes(p)
    extra = {}
    if not args.no_cpu_baseline:
        extra = bwd_cpu_baseline_and_parity(p, g_np, dfin_np, sets[0][0], kernel_name, sets[0][2])
    return {
        **extra,
        "metric": "causal_conv1d_bwd HBM GB/s (x, dout in + dx out bytes) and % of GB300 HBM roofline",
        "value": round(nbytes * args.steps / total_s / 1e9, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": p.name + "_bwd", "io_dtype": p.dtype, "B": p.B, "C": p.C, "L": p.L, "K": p.K,
                   "activation": p.activation or "none", "algorithmic_bytes_per_step": nbytes,
                   "workspace_bytes": sets[0][2], "kernel": kernel_name,
                   "l2": f"inputs larger than L2; {n_sets} rotating buffer sets"},
        "roofline": {"bound": "hbm", "achieved": round(nbytes / mean_step / 1e9, 2), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(nbytes / mean_step / 1e9 / hbm_peak, 4),
                     "traffic": NCU_TRAFFIC.get(kernel_source_hash(), {}).get(p.name + "_bwd"),
                     "peak_source": peak_source, "step_mean_us": round(mean_step * 1e6, 3),
                     "step_bracketed_us": round(bracketed * 1e6, 3), "timing": TIMING_NOTE,
                     "note": "step = gradient kernel + partial-sum reduction kernel; traffic: the gradient kernel's"},
        "gpu_launches": 2 * args.steps, "clocks": clocks,
    }


def bwd_cpu_baseline_and_parity(p, g_np, dfin_np, keep, kernel_name, ws_bytes, budget_s=10.0):
    """Time the oracle's backward single-threaded on the first channels of the
    workload (all b and t; about budget_s of CPU work) and compare the GPU
    gradients of those channels with it under the backward tolerance."""
    import numpy as np
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import compare
    from oracle import oracle as orc

    x = p.x_view()
    dout_v = p._view(g_np, p.x_offset, (p.B, p.C, p.L), p.x_strides)
    init = p.init_view()

    def oracle_channels(lo, hi):
        sl = slice(lo, hi)
        return orc.causal_conv1d_bwd(
            np.ascontiguousarray(x[:, sl, :]), np.ascontiguousarray(p.weight[sl]),
            None if p.bias is None else np.ascontiguousarray(p.bias[sl]), p.dtype,
            np.ascontiguousarray(dout_v[:, sl, :]), p.activation, p.seq_idx,
            None if init is None else np.ascontiguousarray(init[:, sl, :]),
            None if dfin_np is None else np.ascontiguousarray(dfin_np[:, sl, :]), weight_dtype=p.wdt)

    t0 = time.perf_counter()
    oracle_channels(0, 1)
    per_channel = time.perf_counter() - t0
    nc = int(max(1, min(p.C, budget_s / max(per_channel, 1e-9))))
    t0 = time.perf_counter()
    r = oracle_channels(0, nc)
    secs = time.perf_counter() - t0
    sample = bwd_algorithmic_bytes(p) * nc / p.C
    d, gbuf, dfin, dx, dw, db, di, ws = keep
    P = ws_bytes // ((p.K + 1) * p.C * 4) if ws_bytes else 0
    gdw = compare.gamma_dw(kernel_name, p.B, p.L, P)
    checks = [("dx", dv.torch_to_host(dx[:, :nc], p.dtype), r.dx, r.scale["dx"], compare.GAMMA_DX, p.dtype),
              ("dweight", dv.torch_to_host(dw[:nc], p.wdt), r.dweight, r.scale["dweight"], gdw, p.wdt)]
    if db is not None:
        checks.append(("dbias", dv.torch_to_host(db[:nc], p.wdt), r.dbias, r.scale["dbias"], gdw, p.wdt))
    if di is not None:
        checks.append(("dinitial_states", dv.torch_to_host(di[:, :nc], p.dtype), r.dinitial_states,
                       r.scale["dinitial_states"], compare.GAMMA_DX, p.dtype))
    par = {"channels_checked": nc, "tolerance": "|gpu - exact| <= ulp(exact) + gamma * S (oracle/compare.py)"}
    for key, got, exact, scale, gamma, fmt in checks:
        nb, worst, max_ulp = compare.within(got, exact, scale, fmt, gamma)
        par[key] = {"checked": int(exact.size), "outside_tolerance": nb, "max_err_ulp": round(max_ulp, 3),
                    "largest_err_over_bound": round(worst, 4)}
    base = {"value": round(sample / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"channels [0, {nc}) of the workload, all b and t ({nc} of {p.C}), {secs:.1f} s, "
                      "single-threaded C oracle (FP64)",
            "host_cores_available": os.cpu_count(), "host_cpu": host_cpu_model()}
    return {"cpu_baseline": base, "parity_sample": par}


def run_update_bench(args):
    """Decode step (ccv_update) on the bf16 prefill shape's channels: B=8,
    C=5120, S=1, K=4, SiLU.  Reports microseconds per step and the bytes it
    moves (x, out, state read and written, weight, bias); the oracle's step
    on the host is timed beside it and checks one GPU step."""
    import ctypes
    import numpy as np
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding, inputs
    from causal_depthwise_conv1d_gb300 import device as dv

    B, C, S, K, dt = 8, 5120, 1, 4, "bf16"
    rng = np.random.default_rng(0)
    x_np = inputs.round_to_storage(rng.standard_normal(B * C * S), dt).reshape(B, C, S)
    w_np = inputs.round_to_storage(rng.uniform(-0.5, 0.5, C * K), dt).reshape(C, K)
    b_np = inputs.round_to_storage(rng.uniform(-0.5, 0.5, C), dt)
    st_np = inputs.round_to_storage(rng.standard_normal(B * C * (K - 1)), dt).reshape(B, C, K - 1)
    x = dv.host_to_torch(x_np, dt).cuda()
    w = dv.host_to_torch(w_np, dt).cuda()
    b = dv.host_to_torch(b_np, dt).cuda()
    st = dv.host_to_torch(st_np, dt).cuda()
    out = torch.empty_like(x)
    lib = ccv.load_library()
    arr = binding._arr

    def call_for(state, o):
        return (ctypes.c_void_p(x.data_ptr()), arr(x.stride()), ctypes.c_void_p(o.data_ptr()), arr(o.stride()),
                ctypes.c_void_p(state.data_ptr()), arr(state.stride()), ctypes.c_void_p(w.data_ptr()),
                arr(w.stride()), ctypes.c_void_p(b.data_ptr()), ctypes.c_int64(1), ctypes.c_int64(B),
                ctypes.c_int64(C), ctypes.c_int64(S), ctypes.c_int(K), ctypes.c_int(binding.CCV_BF16),
                ctypes.c_int(1), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))

    # one checked step on a copy of the state
    st_chk, out_chk = st.clone(), torch.empty_like(x)
    assert lib.ccv_update(*call_for(st_chk, out_chk)) == 0
    kernel = ccv.ccv_last_kernel()
    call = call_for(st, out)
    for _ in range(args.warmup):
        assert lib.ccv_update(*call) == 0
    torch.cuda.synchronize()
    # timed region: eager steps back to back (each reads the state the
    # previous one wrote), one host launch per step, events at the two ends
    sampler = ClockSampler(smi_index(0))
    sampler.start()
    time.sleep(0.2)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    for _ in range(args.steps):
        lib.ccv_update(*call)
    r1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    per_step = r0.elapsed_time(r1) * 1e3 / args.steps
    # context: the median of steps each between two events of its own
    n_br = min(args.steps, 2000)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_br)]
    for s0, e0 in ev:
        s0.record()
        lib.ccv_update(*call)
        e0.record()
    torch.cuda.synchronize()
    us = sorted(s0.elapsed_time(e0) * 1e3 for s0, e0 in ev)
    med = us[len(us) // 2]
    nbytes = 2 * (2 * B * C * S + 2 * B * C * (K - 1) + C * K + C)
    result = {"metric": "causal_conv1d_update decode step latency", "value": round(per_step, 3), "unit": "us",
              "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
              "dtype": "f32", "data": "synthetic",
              "config": {"workload": "update_bf16_B8_C5120_S1_K4_silu", "io_dtype": dt, "bytes_per_step": nbytes},
              "timing": "eager steps back to back, one host launch each, events at the region's ends",
              "bracketed_median_us": round(med, 3), "gbps": round(nbytes / per_step / 1e3, 1), "kernel": kernel,
              "gpu_launches": args.steps + n_br + 64 * 23, "clocks": clocks}
    # a 64-step decode loop captured once in a CUDA graph and replayed: the
    # per-step cost without a host launch per step
    n_graph = 64
    xs = [x.clone() for _ in range(n_graph)]
    outs = [torch.empty_like(x) for _ in range(n_graph)]
    st_g = st.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for xi, oi in zip(xs, outs):
            ccv.ccv_update(xi, st_g, w, b, activation="silu", out=oi)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    g0.record()
    for _ in range(reps):
        graph.replay()
    g1.record()
    torch.cuda.synchronize()
    result["graph"] = {"value": round(g0.elapsed_time(g1) * 1e3 / (reps * n_graph), 3), "unit": "us per step",
                       "steps_per_graph": n_graph,
                       "note": "decode loop captured once in a CUDA graph and replayed (no host launch per step)"}
    if not args.no_cpu_baseline:
        from oracle import compare
        from oracle import oracle as orc
        t0 = time.perf_counter()
        ref_out, ref_state = orc.causal_conv1d_update(x_np, st_np, w_np, b_np, dt, "silu")
        secs = time.perf_counter() - t0
        rep = compare.compare_out(dv.torch_to_host(out_chk, dt), ref_out, dt)
        result["cpu_baseline"] = {"value": round(secs * 1e6, 1), "unit": "us", "cores": 1, "kind": "oracle",
                                  "sample": "the whole step (8 x 5120 rows), single-threaded C oracle (FP64)",
                                  "host_cores_available": os.cpu_count(), "host_cpu": host_cpu_model()}
        result["parity_sample"] = {"outputs_checked": rep.n, "outside_tolerance": rep.n_bad,
                                   "max_err_ulp": rep.max_err,
                                   "state_bit_exact": compare.compare_bits(dv.torch_to_host(st_chk, dt), ref_state) == 0}
    return result


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--config", default="2", help="workload 1..5, or 'all' (one JSON line each)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="fwd", choices=["fwd", "update", "bwd"],
                    help="fwd: the forward pass (default); update: the decode step; bwd: the backward pass")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-extras", action="store_true",
                    help="time the kernel only: no copy-bandwidth probe, no e2e leg, no CPU baseline "
                         "(for profiler runs)")
    ap.add_argument("--sets", type=int, default=N_SETS, help="rotating device buffer sets")
    ap.add_argument("--no-per-config", action="store_true",
                    help="leave out the per_config record (every workload timed and checked in full)")
    ap.add_argument("--layout", default=None, choices=["interleaved_channel", "interleaved_time"],
                    help="store x of the workload in another layout (same values; neither dimension "
                         "unit-stride), for the strided path")
    return ap


def main():
    ap = build_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    from causal_depthwise_conv1d_gb300 import inputs

    configs = [1, 2, 3, 4, 5] if args.config == "all" else [int(args.config)]
    if args.op == "update":
        if args.impl == "ours" and rank == 0:
            print(json.dumps(run_update_bench(args)), flush=True)
        return
    def workload(idx):
        p = inputs.make_config(idx)
        return inputs.restride(p, args.layout) if args.layout else p

    if args.op == "bwd":
        if args.impl == "ours" and rank == 0:
            for idx in configs:
                print(json.dumps(run_bwd_bench(args, workload(idx), 1, local)), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        for idx in configs:
            print(json.dumps(run_reference(args, workload(idx))), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        for idx in configs:
            p = workload(idx)
            result, out_dev = run_ours(args, p, world, rank, local)
            if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.skip_extras):
                base, par = cpu_baseline_and_parity(p, out_dev)
                result["cpu_baseline"] = base
                result["parity_sample"] = par
            if rank == 0 and world == 1 and args.config != "all" and not (args.skip_extras or args.no_per_config):
                del out_dev
                out_dev = None
                result["per_config"] = per_config_record(local)
                result["per_config_note"] = (
                    "each workload: 2000 back-to-back launches timed like the headline, four rotating buffer "
                    "sets, clocks sampled during that region; every output of the last launch compared with "
                    "the oracle (final_states bit for bit)")
            if rank == 0:
                print(json.dumps(result), flush=True)
            del out_dev
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
