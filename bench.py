#!/usr/bin/env python3
"""Benchmark of the fused selective-scan forward pass on one B300 (plus the decode step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one fused forward pass (discretise, recurrence, read-out, D skip, SiLU gate,
last_state) over the Mamba-1.4B-shaped layer workload: batch 4, L 4096, D 4096, N 16,
bf16 I/O, fp32 state. Inputs (539 MB) are larger than L2 (126 MB), so no flush is
needed between steps. Prints one JSON line (rank 0).

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the
workload shards by batch/channel with no exchange; replicas give weak scaling).

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan fwd GB/s & elem/s (B·L·D) on 1 B300; % of roofline"

# mma.sync m16n8k16 bf16 -> fp32 with independent accumulators, measured on one B300:
# 2048 FLOP/clk/SM; x 148 SMs x 2.032 GHz (the SSD step-size pass's instruction; the
# SSD state walk and read-out run on tcgen05 and are reported against the cuBLAS peak)
MMA_SYNC_TFLOPS = 2048 * 148 * 2.032e9 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "sm_max_mhz": 2032.0, "source": "fallback"}
SM_COUNT = 148
EX2_PER_CLK_SM = 32       # measured on B300: MUFU.EX2 32 lanes/clk/SM
FP32_PER_CLK_SM = 128     # FFMA lanes/clk/SM


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def profiled_traffic():
    """DRAM bytes per forward launch from the committed Nsight Compute summary, or None
    when the kernel's sources have changed since those counters were taken."""
    import re
    prof = os.path.join(ROOT, "profiles", "scan_fwd_chan_m1p4b.md")
    csrc = os.path.join(ROOT, "selective_state_space_141_b300", "csrc")
    srcs = [os.path.join(csrc, f) for f in KERNEL_SOURCES]
    if not (os.path.exists(prof) and all(os.path.exists(f) for f in srcs)):
        return None
    text = open(prof).read()
    t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    if not (t and h):
        return None
    return int(t.group(1)) if kernel_source_hash(srcs) == h.group(1) else None


# The sources the forward kernel is compiled from (its own file and the headers it uses).
KERNEL_SOURCES = ("scan_fwd_chan.cuh", "scan_fwd.cuh", "tma.cuh", "common.cuh")


def kernel_source_hash(paths):
    """First 16 hex digits of the sha256 of the files' bytes, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for f in paths:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def alu_peak_elem_steps(sm_mhz, sms=SM_COUNT):
    """Element-steps/s at the ALU roofline: one ex2 (32/clk/SM) and 4 fp32 ops
    (128/clk/SM) per (b, t, d, n): both pipes give the same bound on B300."""
    return min(sms * EX2_PER_CLK_SM, sms * FP32_PER_CLK_SM / 4) * sm_mhz * 1e6


# ---- clocks ------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        which = "timed region"
        if len(inside) < 3:  # short timed region: fall back to all samples under this run
            inside = [p for (t, p) in self.samples]
            which = "whole run (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        reasons = set()
        for p in inside:
            for name, v in zip(self.NAMES, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][2]),
                "reasons": sorted(reasons), "samples": len(inside), "sampled_over": which,
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


# ---- distributed plumbing (replicas; timing barrier and max only) -------------------------
def dist_init():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle timing -----------------------------------------------------------------
def oracle_sample(w, seconds, seed=0, threads=None):
    """Time the oracle on whole-sequence channels of batch row 0, sized to ~``seconds``, on
    ``threads`` host threads (all CPUs by default).
    Returns (elements (B*L*D units) processed, wall seconds, channels, threads)."""
    import numpy as np
    import torch

    import oracle
    from selective_state_space_141_b300 import inputs

    threads = threads or os.cpu_count() or 1
    g = torch.Generator().manual_seed(seed)
    L, N = w.L, w.N

    def make(k):
        io = w.dtype
        return dict(u=torch.randn(1, L, k, generator=g).to(io), delta=(torch.randn(1, L, k, generator=g) * 0.5 - 2).to(io),
                    z=torch.randn(1, L, k, generator=g).to(io), B=torch.randn(1, L, N, generator=g).to(io),
                    C=torch.randn(1, L, N, generator=g).to(io), D=torch.randn(k, generator=g),
                    delta_bias=(torch.rand(k, generator=g) * (inputs.BIAS_HI - inputs.BIAS_LO) + inputs.BIAS_LO)
                    if w.has_bias else None, A=inputs.s4d_real_A(k, N))

    def run(d):
        arr = {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        t0 = time.perf_counter()
        oracle.selective_scan_fwd(arr["u"], arr["delta"], arr["A"], arr["B"], arr["C"], D=arr["D"], z=arr["z"],
                                  delta_bias=arr["delta_bias"], delta_softplus=True, nthreads=threads)
        return time.perf_counter() - t0

    k0 = min(w.D * w.batch, threads * 32)
    t_cal = run(make(k0))
    k = int(max(k0, min(w.D * w.batch, k0 * seconds / max(t_cal, 1e-3))))
    k = max(threads, (k // threads) * threads)
    t = run(make(k))
    return k * L, t, k, threads


def cpu_model():
    """The host CPU's model name (Linux /proc/cpuinfo), or the platform's processor string."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def cpu_baseline_obj(w, seconds):
    elems, t, k, threads = oracle_sample(w, seconds)
    e1, t1, k1, _ = oracle_sample(w, min(2.0, seconds), threads=1)
    frac = elems / w.elems
    gbs = w.compulsory_bytes() * frac / t / 1e9
    return {"value": gbs, "unit": "GB/s", "elem_per_s": elems / t, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "single_thread": {"elem_per_s": e1 / t1, "GB/s": w.compulsory_bytes() * (e1 / w.elems) / t1 / 1e9,
                              "sample": f"{k1} whole-sequence channels, 1 thread, {t1:.1f} s"},
            "sample": f"{k} whole-sequence channels (L={w.L}, N={w.N}) of batch row 0, fp64, "
                      f"{threads} threads, {t:.1f} s; GB/s scaled by the sample's share of compulsory bytes"}


# ---- the reference arm: the oracle as it stands -------------------------------------------
def run_reference(args, w, ws, rank):
    if rank != 0:
        return
    per_step = max(0.5, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    times, elems = [], 0
    ks = []
    for _ in range(args.steps):
        e, t, k, threads = oracle_sample(w, per_step)
        times.append(t)
        elems += e
        ks.append(k)
    total = sum(times)
    frac = elems / w.elems
    gbs = w.compulsory_bytes() * frac / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "L": w.L, "D": w.D, "N": w.N, "io": "bf16",
                       "sample_per_step": f"~{statistics.median(ks)} whole-sequence channels"},
            "elem_per_s": elems / total,
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
                             "sample": f"each step: whole-sequence channels of one batch row, ~{per_step:.1f} s"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- our arm --------------------------------------------------------------------------
def run_ours(args, w, ws, rank, local):
    import torch

    from selective_state_space_141_b300 import inputs, ssm

    ssm.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    peaks = load_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2032.0))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    alu_peak = alu_peak_elem_steps(sm_max, props.multi_processor_count)

    d = inputs.fwd_inputs(w, dev)
    y = torch.empty_like(d["u"])
    last = torch.empty(w.batch, w.D, w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                               delta_bias=d["delta_bias"], delta_softplus=True, y=y, last_state=last,
                               stream=stream)

    uid = str(getattr(props, "uuid", ""))
    gpu_id = (uid if uid.startswith("GPU-") else "GPU-" + uid) if uid else str(local)
    sampler = ClockSampler(gpu_id)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    h0 = time.time()
    e0.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    barrier(ws)
    total_ms = e0.elapsed_time(e1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(total_ms, ws)
    if ssm.device_error() != 0:
        raise RuntimeError("device error word set during the timed region")
    # the clocks are read over the timed region; extend briefly so short runs still get samples
    if h1 - h0 < 0.5:
        t_end = time.time() + 0.6
        while time.time() < t_end:
            step()
        torch.cuda.synchronize()
        h1 = time.time()
    sampler.stop()
    clocks = sampler.summary(h0, h1)

    sec = total_ms / 1e3
    gbs = ws * K * w.compulsory_bytes() / sec / 1e9
    elem_s = ws * K * w.elems / sec
    achieved = w.element_steps / (launch_ms / 1e3)
    result = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "L": w.L, "D": w.D, "N": w.N, "io": "bf16",
                   "state": "fp32", "l2": "inputs (539 MB) larger than L2 (126 MB); no flush between steps",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "elem_per_s": elem_s,
        "roofline": {
            "bound": "alu", "achieved": achieved / 1e12, "peak": alu_peak / 1e12,
            "unit": "T element-steps/s (1 ex2 + 4 fp32 ops each)", "frac": achieved / alu_peak,
            "traffic": args.traffic if args.traffic is not None else (
                profiled_traffic() if args.workload == "m1p4b" else None),
            "traffic_unit": "bytes per launch (DRAM read + write, Nsight Compute)",
            "algorithmic_bytes": w.compulsory_bytes(),
            "peak_basis": f"{props.multi_processor_count} SMs x 32 ex2/clk (= 128 fp32 lanes / 4 ops) x "
                          f"{sm_max:.0f} MHz max SM clock",
            "launch_ms": launch_ms,
            "hbm": {"achieved_gbs": w.compulsory_bytes() / (launch_ms / 1e3) / 1e9, "peak_gbs": hbm_peak,
                    "frac": w.compulsory_bytes() / (launch_ms / 1e3) / 1e9 / hbm_peak,
                    "peak_source": peaks.get("source")},
        },
        "gpu_launches": K,
        "clocks": clocks,
    }
    if not args.no_e2e:
        result["e2e"] = e2e(w, d, args, ssm, torch, stream)
    if not args.no_decode:
        result["decode"] = decode_bench(args, ssm, torch, inputs, dev, hbm_peak)
    if not args.no_bwd:
        result["backward"] = backward_bench(args, ssm, torch, w, d, dev, launch_ms)
    if not args.no_ssd:
        result["ssd"] = ssd_bench(args, ssm, torch, inputs, dev, peaks)
    samples = {}
    if not args.no_configs:
        result["configs"], samples = configs_bench(args, ssm, torch, inputs, dev, alu_peak, hbm_peak)
        if "decode" in result:
            dec = result["decode"]
            result["configs"]["decode"] = {"workload": dec["workload"], "us_per_step": dec["us_per_step"],
                                           "GB/s": dec["GB/s"], "elem_per_s": dec["elem_per_s"],
                                           "roofline": {"bound": "hbm", "frac": dec["hbm_frac"]}}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_obj(w, args.cpu_seconds)
        if samples:
            # the oracle on the configs' sampled channels: GPU output error from the same run
            for key, e in sampled_oracle_errors(samples).items():
                result["configs"][key]["oracle_check"] = e
    if rank == 0:
        print(json.dumps(result), flush=True)


def configs_bench(args, ssm, torch, inputs, dev, alu_peak, hbm_peak):
    """Every forward workload besides the headline one, each through the plain
    ssm_selective_scan_fwd call (no workspace), and the decode workload: CUDA event time per
    call over calls issued back to back (median of three runs), throughput and both
    roofline terms. Returns (objects, samples):
    samples keep sampled channels' inputs and GPU outputs on the host for the oracle check
    that the CPU-baseline leg runs."""
    import numpy as np

    out, samples = {}, {}
    rng = np.random.default_rng(2024)
    stream = torch.cuda.current_stream()
    for key, reps in (("tiny", 50), ("m130m", 20), ("long", 8)):
        w = inputs.FWD_WORKLOADS[key]
        d = inputs.fwd_inputs(w, dev)
        y = torch.empty_like(d["u"])
        last = torch.empty(w.batch, w.D, w.N, dtype=torch.float32, device=dev)

        def call():
            ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                   delta_bias=d["delta_bias"], delta_softplus=w.delta_softplus, y=y,
                                   last_state=last, stream=stream, use_workspace=False)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        # calls back to back between the events, as the headline's steps: the host's per-call
        # work (argument checks, tensor maps) overlaps the device's
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                call()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / reps)
        if ssm.device_error() != 0:
            raise RuntimeError(f"device error word set during the {key} timing")
        ms = statistics.median(ts)
        t_alu = w.element_steps / alu_peak * 1e3
        t_hbm = w.compulsory_bytes() / (hbm_peak * 1e9) * 1e3
        out[key] = {"workload": w.name, "call": "ssm_selective_scan_fwd (no workspace)", "ms": ms,
                    "GB/s": w.compulsory_bytes() / (ms / 1e3) / 1e9, "elem_per_s": w.elems / (ms / 1e3),
                    "roofline": {"t_alu_ms": t_alu, "t_hbm_ms": t_hbm, "bound": "alu" if t_alu >= t_hbm else "hbm",
                                 "frac": max(t_alu, t_hbm) / ms},
                    "io": "fp32" if w.dtype == torch.float32 else "bf16", "reps": reps,
                    "segmented": ssm.workspace_size(w.batch, w.L, w.D, w.N) > 0 if w.dtype != torch.float32 else None}
        # One more call (untimed) with fp32 output, so the oracle check measures the
        # computation rather than the bf16 output's own rounding.
        if w.dtype != torch.float32:
            y = torch.empty(y.shape, dtype=torch.float32, device=dev)
            call()
            torch.cuda.synchronize()
        b0 = int(rng.integers(w.batch))
        ds = np.sort(rng.choice(w.D, size=min(w.D, 16 if key == "long" else 64), replace=False))
        idx = torch.as_tensor(ds, device=dev)
        pick = lambda t: None if t is None else t[b0:b0 + 1].index_select(2, idx).cpu()
        chan = lambda t: None if t is None else t.index_select(0, idx).cpu()
        samples[key] = dict(u=pick(d["u"]), delta=pick(d["delta"]), z=pick(d["z"]), B=d["B"][b0:b0 + 1].cpu(),
                            C=d["C"][b0:b0 + 1].cpu(), A=chan(d["A"]), D=chan(d["D"]), delta_bias=chan(d["delta_bias"]),
                            delta_softplus=w.delta_softplus, y=pick(y), last=last[b0:b0 + 1].index_select(1, idx).cpu())
        del d, y, last
        torch.cuda.empty_cache()
    return out, samples


def sampled_oracle_errors(samples):
    """Max |GPU - oracle| / rms(oracle) over each config's sampled channels (the oracle fed
    the same inputs), with the oracle's time for the sample."""
    import numpy as np

    import oracle

    res = {}
    for key, sm in samples.items():
        arr = {k: (v.double().numpy() if hasattr(v, "double") else v) for k, v in sm.items()}
        t0 = time.perf_counter()
        yr, sr = oracle.selective_scan_fwd(arr["u"], arr["delta"], arr["A"], arr["B"], arr["C"], D=arr["D"],
                                           z=arr["z"], delta_bias=arr["delta_bias"],
                                           delta_softplus=arr["delta_softplus"], nthreads=os.cpu_count() or 1)
        t = time.perf_counter() - t0
        rms = lambda a: float(np.sqrt(np.mean(a * a)))
        res[key] = {"y_err_rel_rms": float(np.max(np.abs(arr["y"] - yr)) / rms(yr)),
                    "state_err_rel_rms": float(np.max(np.abs(arr["last"] - sr)) / rms(sr)),
                    "channels": int(arr["u"].shape[2]), "oracle_s": t}
    return res


def e2e(w, d, args, ssm, torch, stream):
    """Same metric through the public call with HOST inputs: every step copies its inputs
    from pinned host memory, runs the scan and copies y + last_state back to pinned host
    memory. Steps are pipelined the way a serving loop would run them: two sets of device
    and host buffers, host-to-device copies, the scan and device-to-host copies on three
    streams, so that step i's upload, step i-1's scan and step i-2's download overlap
    (events keep every buffer from being reused before its last reader is done)."""
    names = [k for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias") if d.get(k) is not None]
    host = {k: d[k].cpu().pin_memory() for k in names}
    dev_in = [{k: torch.empty_like(d[k]) for k in names} for _ in range(2)]
    y_h = [torch.empty(d["u"].shape, dtype=d["u"].dtype).pin_memory() for _ in range(2)]
    last_h = [torch.empty(w.batch, w.D, w.N, dtype=torch.float32).pin_memory() for _ in range(2)]
    y = [torch.empty_like(d["u"]) for _ in range(2)]
    last = [torch.empty(w.batch, w.D, w.N, dtype=torch.float32, device=d["u"].device) for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = y_h[0].numel() * y_h[0].element_size() + last_h[0].numel() * 4
    s_in, s_out, s_comp = torch.cuda.Stream(), torch.cuda.Stream(), stream
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    in_done, comp_done, out_done = ev(), ev(), ev()
    used = [False, False]

    def step(i):
        j = i % 2
        if used[j]:
            s_in.wait_event(comp_done[j])  # the scan of step i - 2 has read this input set
            s_comp.wait_event(out_done[j])  # the download of step i - 2 has read this output set
        with torch.cuda.stream(s_in):
            for k in names:
                dev_in[j][k].copy_(host[k], non_blocking=True)
            in_done[j].record(s_in)
        s_comp.wait_event(in_done[j])
        x = dev_in[j]
        ssm.selective_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x.get("D"), z=x.get("z"),
                               delta_bias=x.get("delta_bias"), y=y[j], last_state=last[j], stream=s_comp)
        comp_done[j].record(s_comp)
        s_out.wait_event(comp_done[j])
        with torch.cuda.stream(s_out):
            y_h[j].copy_(y[j], non_blocking=True)
            last_h[j].copy_(last[j], non_blocking=True)
            out_done[j].record(s_out)
        used[j] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_comp.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(n):
        step(2 + i)
    e1.record(s_out)
    torch.cuda.synchronize()
    jl = (2 + n - 1) % 2  # the last step's buffers: the download must equal the device result
    if not (torch.equal(y_h[jl], y[jl].cpu()) and torch.equal(last_h[jl], last[jl].cpu())):
        raise RuntimeError("e2e: downloaded result differs from the device result")
    sec = e0.elapsed_time(e1) / 1e3 / n
    return {"value": w.compulsory_bytes() / sec / 1e9, "unit": "GB/s", "ms_per_step": sec * 1e3,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "pipelining": "2 buffer sets; uploads, scans and downloads on 3 streams"}


def backward_bench(args, ssm, torch, w, d, dev, fwd_launch_ms):
    """The backward pass (all gradients) on the same workload, bf16 dy, CUDA events around
    each call. Standalone (`ms`): three launches, the checkpoint pass (the channel kernel's
    recurrence without read-out), the reverse kernel and the fixed-order reduction. In a
    training step (`training_step`): the forward pass writes the checkpoints itself
    (ssm_selective_scan_fwd_train) and the backward pass is the last two launches."""
    g = torch.Generator(device=dev).manual_seed(5)
    dy = torch.randn(d["u"].shape, generator=g, device=dev).to(d["u"].dtype)
    nbytes = ssm.bwd_workspace_size(w.batch, w.L, w.D, w.N)
    wsp = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    y = torch.empty(d["u"].shape, dtype=d["u"].dtype, device=dev)
    last = torch.empty((w.batch, w.D, w.N), dtype=torch.float32, device=dev)
    written = [False]

    def bwd(ready=False):
        return ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], dy, D=d["D"], z=d["z"],
                                      delta_bias=d["delta_bias"], delta_softplus=True, workspace=wsp,
                                      checkpoints_ready=ready)

    def fwd_train():
        written[0] = ssm.selective_scan_fwd_train(d["u"], d["delta"], d["A"], d["B"], d["C"], wsp, D=d["D"], z=d["z"],
                                                  delta_bias=d["delta_bias"], delta_softplus=True, y=y,
                                                  last_state=last)[2]

    # Calls are issued back to back between the events (as the forward pass's steps are),
    # so the host's per-call work (argument checks, tensor maps) overlaps the GPU's instead
    # of being counted as device time.
    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.bwd_steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.bwd_steps

    m = timed(bwd)
    # training step: the forward pass with checkpoints, then the backward pass that uses them
    mf = timed(fwd_train)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.bwd_steps + 1)]
    for i in range(args.bwd_steps):  # back to back: forward, backward, forward, ...
        ev[2 * i].record()
        fwd_train()
        ev[2 * i + 1].record()
        bwd(ready=written[0])
    ev[2 * args.bwd_steps].record()
    torch.cuda.synchronize()
    mfb = [ev[2 * i].elapsed_time(ev[2 * i + 2]) for i in range(args.bwd_steps)]
    mb = [ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(args.bwd_steps)]
    if ssm.device_error() != 0:
        raise RuntimeError("device error word set during the backward pass")
    mb_med = statistics.median(mb)
    return {"workload": w.name, "ms": m, "ratio_to_forward": m / fwd_launch_ms, "elem_per_s": w.elems / (m / 1e3),
            "calls": args.bwd_steps, "workspace_bytes": nbytes, "launches_per_call": 3,
            "gradients": "du, ddelta, dA, dB, dC, dD, dz, dbias (bf16 dy; fp32 accumulation)",
            "training_step": {"forward_with_checkpoints_ms": mf, "backward_ms": mb_med,
                              "backward_ratio_to_forward": mb_med / fwd_launch_ms,
                              "forward_plus_backward_ms": statistics.median(mfb),
                              "checkpoints_written": bool(written[0]), "backward_launches": 2}}


def ssd_bench(args, ssm, torch, inputs, dev, peaks):
    """The Mamba-2 SSD workload (chunked, tensor cores): CUDA events around one replay of a
    CUDA graph of back-to-back calls."""
    w = inputs.SSD_M2
    d = inputs.ssd_inputs(w, dev)
    y = torch.empty_like(d["x"])
    ls = torch.empty(w.batch, w.H, w.P, w.N, dtype=torch.float32, device=dev)
    nbytes = ssm.ssd_workspace_size(w.batch, w.L, w.H, w.P, w.N, groups=w.G)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def call():
        ssm.ssd_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], dt_bias=d["dt_bias"], dt_softplus=True,
                    y=y, last_state=ls, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # the calls captured in one CUDA graph, so that the binding's host work per call (about
    # as long as the call's device time here) stays off the device timeline
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(args.ssd_steps):
            call()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    if ssm.device_error() != 0:
        raise RuntimeError("device error word set during the SSD calls")
    m = e0.elapsed_time(e1) / args.ssd_steps
    tf = w.flops() / (m / 1e3) / 1e12
    tpk = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    gbs = w.compulsory_bytes() / (m / 1e3) / 1e9
    hpk = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": w.name, "ms": m, "tokens_per_s": w.tokens / (m / 1e3),
            "roofline": {"bound": "tensor" if w.flops() / (tpk * 1e12) > w.compulsory_bytes() / (hpk * 1e9) else "hbm",
                         "tensor": {"achieved": tf, "peak": tpk, "unit": "TFLOP/s", "frac": tf / tpk,
                                    "flops_per_call": w.flops(),
                                    "mma_sync_peak": MMA_SYNC_TFLOPS, "frac_of_mma_sync": tf / MMA_SYNC_TFLOPS},
                         "hbm": {"achieved_gbs": gbs, "peak_gbs": hpk, "frac": gbs / hpk,
                                 "algorithmic_bytes": w.compulsory_bytes()}},
            "calls": args.ssd_steps, "timing": "one CUDA graph of the calls", "workspace_bytes": nbytes,
            "launches_per_call": 3,
            "kernel": "step sizes + C B^T per chunk (mma.sync); state walk and persistent read-out on tcgen05 "
                      "(TMEM accumulators, TMA operands, warp-specialised copier / MMA / worker warps); bf16 "
                      "operands (hi/lo pairs for products of inputs), fp32 accumulate"}


def decode_bench(args, ssm, torch, inputs, dev, hbm_peak, layers=4):
    """The decode workload: 1024 single-token steps captured in one CUDA graph. The steps
    cycle over `layers` layer states (as a model steps through its layers for each token),
    so the states together (4 x 84 MB) exceed L2 and every step reads its state from HBM."""
    w = inputs.DECODE
    T = args.decode_steps
    d = inputs.decode_inputs(w, dev, steps=T)
    ys = torch.empty(T, w.batch, w.D, dtype=w.dtype, device=dev)
    states = [d["state"].clone() for _ in range(layers)]

    def step(t):
        ssm.state_update(states[t % layers], d["x"][t], d["delta"][t], d["A"], d["B"][t], d["C"][t], D=d["D"],
                         z=d["z"][t], y=ys[t])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        for t in range(2):
            step(t)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for t in range(T):
            step(t)
    g.replay()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    if ssm.device_error() != 0:
        raise RuntimeError("device error word set during decode")
    per_step = e0.elapsed_time(e1) / 1e3 / (reps * T)
    bps = w.bytes_per_step()
    state_mb = states[0].numel() * 4 / 1e6
    return {"workload": w.name, "us_per_step": per_step * 1e6, "GB/s": bps / per_step / 1e9,
            "hbm_frac": bps / per_step / 1e9 / hbm_peak, "bytes_per_step": bps, "steps_per_graph": T,
            "elem_per_s": w.batch * w.D / per_step, "layer_states": layers,
            "note": f"steps cycle over {layers} layer states ({layers} x {state_mb:.0f} MB, more than the "
                    "126 MB L2), so each step streams its state from HBM; GB/s counts compulsory bytes per step"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="m1p4b")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--bwd-steps", type=int, default=5)
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--ssd-steps", type=int, default=10)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel (else null)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from selective_state_space_141_b300 import inputs
    w = inputs.FWD_WORKLOADS[args.workload]
    ws, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, w, ws, rank)
    else:
        run_ours(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
