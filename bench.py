#!/usr/bin/env python3
"""Benchmark of the selective-scan forward (libselscan) on B300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one ``selscan_fwd`` over one batch of the workload: softplus Δ,
discretisation, the chunked scan, the C readout, the D skip and the SiLU gate
(every row of the forward hot path), with inputs resident in HBM.  The default
workload is the Mamba-130M-like layer scan (batch 8, d_inner 1536, L 2048,
d_state 16, bf16 u/δ/z/B/C, fp32 state and fp32 out).  L2 is flushed (a
256 MiB write) before every timed step, outside the step's CUDA events.

Reported: ``value`` = elements (B·D·L) per second over all GPUs, from the
per-step CUDA-event times summed over the K timed steps (max over ranks);
``hbm_gbs`` = algorithmic bytes / time; ``roofline`` for the fused forward
kernel; ``e2e`` = the same metric with host (pinned) inputs copied in and the
output copied back for every step inside the timed region (steps pipelined
over three streams: copies in, scan, copies out); ``cpu_baseline`` = the fp64 oracle
on the host cores on a bounded row sample; ``decode`` = the recurrent decode
step workload (secondary).  Under torchrun (N > 1) every rank runs its own
shard of an N-times-larger batch (weak scaling, no data-path collective).
``sweep`` times the other forward workloads of the same family (the 65536-step
sequence and the 2.8B-width layer) the same way, each with its own roofline;
``unit_rates`` are the special-function and FMA rates measured on the GPU by the
library's own probe (selscan_probe_rate), from which the rooflines are derived.
``backward`` times selscan_bwd (every gradient, bf16 dout) on the same workloads,
each against the backward's own roofline (``bwd_work``), and the training pair
selscan_fwd_ckpt + selscan_bwd_ckpt (the backward rerunning from the forward's
chunk checkpoints).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "selective-scan elems(B·D·L)/s and HBM GB/s at 1 B300; fraction of roofline"
DEFAULT_WORKLOAD = "mamba130m_layer"
L2_FLUSH_BYTES = 256 << 20
# Results per clock per SM of the units the forward needs, used only when the probe cannot run (no GPU):
# the values selscan_probe_rate measured on B300 (ex2 32; lg2 and rcp at half that rate; fp32 FMA 128).
FALLBACK_RATES = {"ex2": 32.0, "lg2": 16.0, "rcp": 16.0, "ffma2": 128.0}
FALLBACK_HBM_GBS = 6400.0
FALLBACK_SM_MHZ = 2032.0


# ------------------------------------------------------------------------------------------------
# Host-side logic (unit-tested on CPU)
# ------------------------------------------------------------------------------------------------

def measured_peaks(path=os.path.join(ROOT, "MEASURED_PEAKS.json")):
    """(hbm GB/s, max SM MHz, source) from the measured-peaks file beside this script, else the fallback."""
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("sm_max_mhz", FALLBACK_SM_MHZ)), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, FALLBACK_SM_MHZ, "fallback"


def fwd_work(batch, dim, seqlen, dstate, in_bytes=2, out_bytes=4, h0=False, h_last=True):
    """Algorithmic work of one selscan_fwd: elements, bytes, special-function ops and FP32 ops.

    Bytes: u, δ, z read once and out written once per element; B, C read once
    per (b, n, t) — not per channel; A, D, Δ_bias once; h0 / h_last once.
    Special functions per element: N exponentials for Ā, an exponential and a
    logarithm for softplus, an exponential and a reciprocal for the gate
    ("ex2": N + 2, "lg2": 1, "rcp": 1).  FP32: 4 per (element, state) — Δ·A,
    Δu·B, the state FMA, the C·h FMA — plus 8 per element.
    """
    elems = batch * dim * seqlen
    nbytes = elems * (3 * in_bytes + out_bytes) + 2 * batch * dstate * seqlen * in_bytes + dim * dstate * 4 + 2 * dim * 4
    if h0:
        nbytes += batch * dim * dstate * 4
    if h_last:
        nbytes += batch * dim * dstate * 4
    return {"elements": elems, "bytes": nbytes, "mufu": elems * (dstate + 4),
            "sfu": {"ex2": elems * (dstate + 2), "lg2": elems, "rcp": elems}, "fp32": elems * (4 * dstate + 8)}


def bwd_work(batch, dim, seqlen, dstate, in_bytes=2, dout_bytes=2):
    """Algorithmic work of one selscan_bwd (gradients of every input of the forward).

    Bytes: u, δ, z, dout read once and du, dδ, dz written once per element; B, C read and dB, dC
    written once per (b, n, t); A, D, Δ_bias, h0, dh_last, dA, dD, dΔ_bias, dh0 once (the checkpoint
    workspace is not algorithmic).  Special functions per element: the states recomputed once and
    undone once (2N exponentials), softplus (an exponential and a logarithm) whose exponential also
    gives σ(δ + Δ_bias) with one reciprocal, and σ(z) (an exponential and a reciprocal).  FP32: 4 per
    (element, state) for the recomputation, 9 for the reverse sweep, plus 30 per element.
    """
    elems = batch * dim * seqlen
    bc = batch * dstate * seqlen
    nbytes = (elems * (6 * in_bytes + dout_bytes) + bc * (2 * in_bytes + 2 * 4) + 2 * dim * dstate * 4
              + 4 * dim * 4 + 3 * batch * dim * dstate * 4)
    return {"elements": elems, "bytes": nbytes,
            "sfu": {"ex2": elems * (2 * dstate + 2), "lg2": elems, "rcp": 2 * elems},
            "fp32": elems * (13 * dstate + 30)}


def step_work(batch, dim, dstate, in_bytes=2, out_bytes=4):
    """Algorithmic bytes of one decode step: state read + write, u/δ/z/out, B/C, A/D/bias."""
    rows = batch * dim
    return {"elements": rows,
            "bytes": rows * (2 * dstate * 4 + 3 * in_bytes + out_bytes) + 2 * batch * dstate * in_bytes
            + dim * dstate * 4 + 2 * dim * 4}


def mufu_slots(work, rates):
    """Special-function work in ex2-equivalent issue slots: each unit's ops scaled by ex2's rate over its own."""
    sfu = work.get("sfu") or {"ex2": work["mufu"]}
    return sum(n * rates["ex2"] / rates[u] for u, n in sfu.items())


def roofline_times(work, sms, hbm_gbs, sm_mhz, rates=None):
    """Seconds each resource needs at its peak: HBM bytes, special-function ops (each unit at its measured
    rate), FP32 ops."""
    rates = rates or FALLBACK_RATES
    f = sm_mhz * 1e6
    return {"hbm": work["bytes"] / (hbm_gbs * 1e9), "mufu": mufu_slots(work, rates) / (sms * rates["ex2"] * f),
            "fp32": work["fp32"] / (sms * rates["ffma2"] * f)}


def roofline_entry(work, t_kernel, sms, hbm_gbs, sm_mhz, traffic=None, rates=None):
    """The roofline object for a forward kernel that took t_kernel seconds per launch."""
    rates = rates or FALLBACK_RATES
    t = roofline_times(work, sms, hbm_gbs, sm_mhz, rates)
    bound = max(t, key=t.get)
    if bound == "hbm":
        achieved, peak, unit = work["bytes"] / t_kernel / 1e9, hbm_gbs, "GB/s"
        kind = "hbm"
    elif bound == "mufu":
        achieved = mufu_slots(work, rates) / t_kernel / 1e12
        peak = sms * rates["ex2"] * sm_mhz * 1e6 / 1e12
        unit, kind = "TFLOP/s", "alu"
    else:
        achieved = work["fp32"] / t_kernel / 1e12
        peak = sms * rates["ffma2"] * sm_mhz * 1e6 / 1e12
        unit, kind = "TFLOP/s", "alu"
    return {"bound": kind, "resource": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "t_us": {k: v * 1e6 for k, v in t.items()}, "t_kernel_us": t_kernel * 1e6}


def shard_batch(global_batch, rank, world):
    """Contiguous batch range [lo, hi) of this rank (weak scaling: each rank gets global_batch / world)."""
    per = global_batch // world
    rem = global_batch % world
    lo = rank * per + min(rank, rem)
    return lo, lo + per + (1 if rank < rem else 0)


def aggregate(elements_per_rank, seconds_per_rank):
    """Whole-job throughput: all ranks' elements over the slowest rank's time."""
    return sum(elements_per_rank) / max(seconds_per_rank)


def max_over_ranks(seconds, dist, device):
    """The largest of the ranks' times (the job's time); the value itself when not distributed."""
    if dist is None:
        return seconds
    import torch

    tt = torch.tensor([float(seconds)], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


# The sources each measured kernel is built from (its own file and the shared device helpers): the forward
# workloads run the row-sequential kernel.
KERNEL_SOURCES = {"selscan_fwd": ("selscan_rows.cu", "selscan_internal.cuh"),
                  "selscan_step": ("selscan_step.cu", "selscan_internal.cuh"),
                  "selscan_bwd": ("selscan_bwd.cu", "selscan_internal.cuh")}


def kernel_source_hash(kernel=None):
    """Hash of a kernel's sources (all of csrc/ when kernel is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_152_b300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh"))]
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, path=os.path.join(ROOT, "profiles", "ncu_traffic.json")):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel sources."""
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the benchmark runs.

    Sampling starts before the warm-up (``start``, which waits for the first sample: nvidia-smi takes
    a moment to begin) and stops after the run; ``mark_begin`` / ``mark_end`` bracket the timed region
    and ``report`` keeps the samples taken inside it.  NVML is used where importable, else nvidia-smi
    polling.
    """

    REASONS = {"hw_slowdown": "nvmlClocksEventReasonHwSlowdown",
               "hw_thermal_slowdown": "nvmlClocksEventReasonHwThermalSlowdown",
               "sw_thermal_slowdown": "nvmlClocksEventReasonSwThermalSlowdown",
               "sw_power_cap": "nvmlClocksEventReasonSwPowerCap",
               "hw_power_brake": "nvmlClocksEventReasonHwPowerBrakeSlowdown"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
    SMI_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index, period_s=0.02, smi_id=None):
        self.samples = []  # (time, sm MHz, set of active reasons)
        self.max_mhz, self.error = None, None
        self.smi_id = smi_id if smi_id is not None else str(device_index)
        self.period = period_s
        self.begin = self.end = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        try:
            import pynvml

            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception as e:  # noqa: BLE001 - fall back to nvidia-smi polling
            self.nv = None
            self.error = f"{type(e).__name__}: {e}"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                reasons = {name for name, const in self.REASONS.items() if r & getattr(nv, const, 0)}
                self.samples.append((time.perf_counter(), float(mhz), reasons))
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def _run_smi(self):
        for line in self._proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 6:
                continue
            try:
                mhz = float(f[0])
                self.max_mhz = float(f[1])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.SMI_NAMES, f[2:6]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), mhz, reasons))

    def start(self, wait_s=5.0):
        if self.nv is not None:
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
        else:
            import subprocess

            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", str(max(20, int(self.period * 1000))), "-i", self.smi_id],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            except OSError as e:
                self.error = (self.error or "") + f"; nvidia-smi: {e}"
                return self
            self._t = threading.Thread(target=self._run_smi, daemon=True)
        self._t.start()
        t0 = time.perf_counter()
        while not self.samples and time.perf_counter() - t0 < wait_s:
            time.sleep(0.01)
        return self

    def mark_begin(self):
        self.begin = time.perf_counter()

    def mark_end(self):
        self.end = time.perf_counter()

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=10)
            except Exception:  # noqa: BLE001
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=10)

    def report(self):
        lo = self.begin if self.begin is not None else -float("inf")
        hi = self.end if self.end is not None else float("inf")
        inside = [(mhz, rs) for t, mhz, rs in self.samples if lo <= t <= hi]
        reasons = set().union(*[rs for _, rs in inside]) if inside else set()
        r = {"sm_mhz": statistics.median([m for m, _ in inside]) if inside else None, "sm_max_mhz": self.max_mhz,
             "reasons": sorted(reasons), "samples": len(inside), "samples_total": len(self.samples),
             "timed_region_s": (hi - lo) if self.begin is not None and self.end is not None else None,
             "source": "nvml" if self.nv is not None else "nvidia-smi"}
        if self.error:
            r["nvml_error"] = self.error
        return r


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------

def _dev(torch, a, device):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def _pinned(torch, a):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(a).pin_memory()


def workload_config(w, batch, seqlen):
    """The `config` object of a bench line (both arms print the same one)."""
    return {"workload": w.name, "batch": batch, "dim": w.dim, "seqlen": seqlen, "dstate": w.dstate,
            "in_dtype": w.in_dtype, "out_dtype": "f32", "state": "f32",
            "l2": "flushed (256 MiB write) before every timed step, outside its events"}


def measure_rates(ss):
    """The special-function and FMA rates of this GPU (results per clock per SM) from the library's probe."""
    try:
        return {u: ss.selscan_probe_rate(u) for u in ("ex2", "lg2", "rcp", "ffma2")}, "measured (selscan_probe_rate)"
    except Exception as e:  # noqa: BLE001
        return dict(FALLBACK_RATES), f"fallback ({type(e).__name__})"


def time_forward(torch, fwd, stream, flush, steps):
    """CUDA-event time of each of `steps` calls, each after an L2 flush outside its events."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        fwd()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1e3 for a, b in zip(starts, ends)]


def forward_tensors(torch, inp, w, device):
    t = {k: _dev(torch, inp.get(k), device) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    Bsz, Dm, L, N = inp["shape"]
    out = torch.empty((Bsz, Dm, L), device=device, dtype=torch.float32)
    h_last = torch.empty((Bsz, Dm, N), device=device, dtype=torch.float32) if w.returns_h_last else None
    return t, out, h_last


def run_ours(args, rank, world, local_rank, dist):
    import torch

    import selective_state_space_152_b300 as ss

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    w = si.WORKLOADS[args.workload]
    if w.steps:
        raise SystemExit("the timed step is the forward scan; the decode workload is reported under 'decode'")
    lo, hi = shard_batch(w.batch * world, rank, world)
    inp = si.make_inputs(w, seed=si.BASE_SEED + si.WORKLOAD_ORDER.index(w.name) + 1000 * rank, batch=hi - lo)
    Bsz, Dm, L, N = inp["shape"]
    t, out, h_last = forward_tensors(torch, inp, w, device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=device, dtype=torch.float32)
    stream = torch.cuda.current_stream()
    rates, rates_src = measure_rates(ss)

    def fwd():
        ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], delta_bias=t["delta_bias"],
                       delta_softplus=True, h0=t["h0"], out=out, h_last=h_last, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    props = torch.cuda.get_device_properties(device)
    smi_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local_rank)
    clk = ClockSampler(local_rank, smi_id=smi_id).start()
    for _ in range(args.warmup):
        flush.zero_()
        fwd()
    launches_per_call = ss.selscan_last_launch_count()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk.mark_begin()
    wall0 = time.perf_counter()
    step_s = time_forward(torch, fwd, stream, flush, args.steps)
    wall = time.perf_counter() - wall0
    clk.mark_end()
    barrier()
    torch.cuda.synchronize()
    t_sum = sum(step_s)
    t_max = max_over_ranks(t_sum, dist, device)
    elems_rank = Bsz * Dm * L * args.steps
    value = elems_rank * world / t_max

    work = fwd_work(Bsz, Dm, L, N, in_bytes=2 if w.in_dtype == "bf16" else 4, out_bytes=4,
                    h0=inp.get("h0") is not None, h_last=h_last is not None)
    sms = props.multi_processor_count
    hbm_gbs, sm_mhz, peak_src = measured_peaks()
    t_kernel = t_sum / args.steps
    roof = roofline_entry(work, t_kernel, sms, hbm_gbs, sm_mhz, rates=rates,
                          traffic=recorded_traffic("selscan_fwd", args.workload))
    roof["peak_source"] = (f"HBM {hbm_gbs} GB/s ({peak_src} copy bandwidth); special-function and FMA rates "
                           f"{rates_src}; SM {sm_mhz} MHz x {sms} SMs")

    result = {
        "metric": METRIC, "value": value, "unit": "elems/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, Bsz * world, L),
        "hbm_gbs": work["bytes"] * world * args.steps / t_max / 1e9,
        "roofline": roof,
        "gpu_launches": args.steps * launches_per_call,
        "unit_rates": dict(rates, source=rates_src, unit="results per clock per SM"),
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_sweep:
        result["sweep"] = run_sweep(args, torch, ss, device, stream, flush, sms, hbm_gbs, sm_mhz, rates)
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, torch, ss, inp, w, device, stream, flush, dist, world)
    if rank == 0 and world == 1 and not args.no_decode:
        result["decode"] = run_decode(args, torch, ss, device, stream, flush, sms, hbm_gbs)
    if rank == 0 and world == 1 and not args.no_options:
        result["options"] = run_options(ss, torch, t, out, h_last, stream, flush, work, sms, hbm_gbs, sm_mhz, rates)
    if rank == 0 and world == 1 and not args.no_backward:
        result["backward"] = run_backward(args, torch, ss, device, stream, flush, sms, hbm_gbs, sm_mhz, rates)
    clk.stop()
    result["clocks"] = clk.report()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, w, budget_cpu_s=args.cpu_budget)
    return result


SWEEP_WORKLOADS = ("mamba130m_layer", "long_seq_65k", "width_2p8b")


def run_sweep(args, torch, ss, device, stream, flush, sms, hbm_gbs, sm_mhz, rates):
    """Every forward workload of the family timed like the headline (CUDA events per call, L2 flushed
    before each), each against its own roofline."""
    res = {}
    for name in SWEEP_WORKLOADS:
        w = si.WORKLOADS[name]
        inp = si.make_inputs(w)
        Bsz, Dm, L, N = inp["shape"]
        t, out, h_last = forward_tensors(torch, inp, w, device)

        def fwd():
            ss.selscan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], delta_softplus=True, h0=t["h0"], out=out, h_last=h_last,
                           stream=stream)

        for _ in range(3):
            flush.zero_()
            fwd()
        launches = ss.selscan_last_launch_count()
        steps = max(5, args.sweep_steps)
        secs = time_forward(torch, fwd, stream, flush, steps)
        t_call = statistics.median(secs)
        work = fwd_work(Bsz, Dm, L, N, in_bytes=2 if w.in_dtype == "bf16" else 4, out_bytes=4,
                        h0=inp.get("h0") is not None, h_last=h_last is not None)
        roof = roofline_entry(work, t_call, sms, hbm_gbs, sm_mhz, rates=rates,
                              traffic=recorded_traffic("selscan_fwd", name))
        res[name] = {"config": workload_config(w, Bsz, L), "steps": steps, "us_per_call": t_call * 1e6,
                     "us_per_call_min": min(secs) * 1e6, "elems_per_s": work["elements"] / t_call,
                     "hbm_gbs": work["bytes"] / t_call / 1e9, "roofline": roof, "launches_per_call": launches}
        del t, out, h_last
        torch.cuda.empty_cache()
    return res


def run_e2e(args, torch, ss, inp, w, device, stream, flush, dist, world):
    """The same metric through the public API with pinned host buffers copied in and out each step.

    Steps are pipelined the way a stream of batches would be: the host->device copies of step k+1
    (one stream), the scan of step k (the compute stream) and the device->host copies of step k-1
    (a third stream) overlap, with two sets of device buffers ordered by events.  Every step still
    moves its full inputs in and its full outputs out.
    """
    Bsz, Dm, L, N = inp["shape"]
    names = ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")
    host = {k: _pinned(torch, inp.get(k)) for k in names}
    sets = [{k: (None if host[k] is None else torch.empty_like(host[k], device=device)) for k in names}
            for _ in range(2)]
    outs = [torch.empty((Bsz, Dm, L), device=device, dtype=torch.float32) for _ in range(2)]
    hls = [torch.empty((Bsz, Dm, N), device=device, dtype=torch.float32) if w.returns_h_last else None
           for _ in range(2)]
    out_h = torch.empty((Bsz, Dm, L), dtype=torch.float32).pin_memory()
    hl_h = torch.empty((Bsz, Dm, N), dtype=torch.float32).pin_memory() if w.returns_h_last else None
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = out_h.numel() * 4 + (hl_h.numel() * 4 if hl_h is not None else 0)
    steps = max(3, min(args.steps, args.e2e_steps))
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in comp_done + out_done:
        e.record(stream)  # nothing outstanding at the start

    def one(j):
        k = j % 2
        dev, out, hl = sets[k], outs[k], hls[k]
        s_in.wait_event(comp_done[k])  # step j-2 has finished reading this input set
        with torch.cuda.stream(s_in):
            for n in names:
                if host[n] is not None:
                    dev[n].copy_(host[n], non_blocking=True)
        in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        stream.wait_event(out_done[k])  # step j-2's outputs have left this output set
        ss.selscan_fwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], D=dev["D"], z=dev["z"],
                       delta_bias=dev["delta_bias"], h0=dev["h0"], out=out, h_last=hl, stream=stream)
        comp_done[k].record(stream)
        s_out.wait_event(comp_done[k])
        with torch.cuda.stream(s_out):
            out_h.copy_(out, non_blocking=True)
            if hl is not None:
                hl_h.copy_(hl, non_blocking=True)
        out_done[k].record(s_out)

    for j in range(2):
        one(j)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    s_in.wait_event(ev0)
    for j in range(steps):
        one(j)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    ev1.record(stream)
    torch.cuda.synchronize()
    secs = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, dist, device)

    # The host link's bound for the same bytes: the same copies on the same streams with no scan.
    def copies(k):
        with torch.cuda.stream(s_in):
            for n in names:
                if host[n] is not None:
                    sets[k][n].copy_(host[n], non_blocking=True)
        with torch.cuda.stream(s_out):
            out_h.copy_(outs[k], non_blocking=True)
            if hls[k] is not None:
                hl_h.copy_(hls[k], non_blocking=True)

    copies(0)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    s_in.wait_event(c0)
    s_out.wait_event(c0)
    for j in range(steps):
        copies(j % 2)
    stream.wait_stream(s_out)
    stream.wait_stream(s_in)
    c1.record(stream)
    torch.cuda.synchronize()
    link = max_over_ranks(c0.elapsed_time(c1) / 1e3, dist, device)
    return {"value": Bsz * Dm * L * steps * world / secs, "unit": "elems/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": secs / steps * 1e3,
            "gpu_launches": steps, "pipelined": "h2d / scan / d2h on three streams, two buffer sets",
            "link_bound": {"ms_per_step": link / steps * 1e3, "frac": link / secs,
                           "what": "the same host copies on the same streams without the scan (pinned memory)"}}


def run_options(ss, torch, t, out, h_last, stream, flush, work, sms, hbm_gbs, sm_mhz, rates, steps=50):
    """Secondary: the options on the same workload (selscan_fwd_ex's reverse scan and exact
    zero-order-hold input matrix; selscan_fwd_conv's conv1d + SiLU front), each call timed after an
    L2 flush, against the same roofline."""
    res = {}
    g = torch.Generator(device="cpu").manual_seed(5)
    Dm = t["A"].shape[0]
    conv_w = (torch.randn((Dm, 4), generator=g) * 0.5).to(t["A"].device)
    conv_b = (torch.randn((Dm,), generator=g) * 0.5).to(t["A"].device)
    for name, kw in (("reverse", dict(reverse=True)), ("zoh", dict(zoh=True)), ("conv", None)):
        def call(kw=kw):
            if kw is None:  # the causal conv1d + SiLU front computed in the kernel (u is read as x)
                ss.selscan_fwd_conv(t["u"], conv_w, conv_b, t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                    delta_bias=t["delta_bias"], delta_softplus=True, h0=t["h0"], out=out,
                                    h_last=h_last, stream=stream)
                return
            ss.selscan_fwd_ex(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                              delta_bias=t["delta_bias"], delta_softplus=True, h0=t["h0"], out=out, h_last=h_last,
                              stream=stream, **kw)

        for _ in range(3):
            flush.zero_()
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        secs = sum(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3 / steps
        roof = roofline_entry(work, secs, sms, hbm_gbs, sm_mhz, rates=rates)
        res[name] = {"us_per_call": secs * 1e6, "elems_per_s": work["elements"] / secs,
                     "roofline_frac": roof["frac"], "gpu_launches": steps}
    return res


BACKWARD_WORKLOADS = ("mamba130m_layer", "width_2p8b", "long_seq_65k")


def run_backward(args, torch, ss, device, stream, flush, sms, hbm_gbs, sm_mhz, rates):
    """Secondary: the backward (selscan_bwd, every gradient) on the forward workloads, each call timed after
    an L2 flush with its workspace allocated beforehand, against the backward's own roofline."""
    res = {}
    for name in BACKWARD_WORKLOADS:
        w = si.WORKLOADS[name]
        inp = si.make_inputs(w)
        Bsz, Dm, L, N = inp["shape"]
        t, _, _ = forward_tensors(torch, inp, w, device)
        cot = si.random_cotangents(77, Bsz, Dm, L, N, dout_dtype="bf16")
        go, gh = _dev(torch, cot["dout"], device), _dev(torch, cot["dh_last"], device)
        ws = torch.empty(ss.selscan_bwd_workspace_size(Bsz, Dm, L, N), dtype=torch.uint8, device=device)
        g = ss.selscan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], go, D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], h0=t["h0"], dh_last=gh, workspace=ws, stream=stream)

        def call():
            ss.selscan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], go, D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], h0=t["h0"], dh_last=gh, grads=g, workspace=ws, stream=stream)

        for _ in range(3):
            flush.zero_()
            call()
        launches = ss.selscan_last_launch_count()
        reps = 5 if L > 10000 else 20
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        secs = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3
        # The training pair: the forward keeping its chunk checkpoints, and the backward rerunning from them.
        out = torch.empty((Bsz, Dm, L), device=device, dtype=torch.float32)
        ck = torch.empty((Bsz, Dm, (L + 15) // 16, 16), device=device, dtype=torch.float32)

        def fwd_ckpt():
            ss.selscan_fwd_ckpt(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                delta_bias=t["delta_bias"], h0=t["h0"], out=out, ckpt=ck, stream=stream)

        def bwd_ckpt():
            ss.selscan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], go, D=t["D"], z=t["z"],
                           delta_bias=t["delta_bias"], h0=t["h0"], dh_last=gh, grads=g, workspace=ws, ckpt=ck,
                           stream=stream)

        pair = {}
        for key, fn in (("fwd_ckpt_us", fwd_ckpt), ("bwd_from_ckpt_us", bwd_ckpt)):
            for _ in range(3):
                flush.zero_()
                fn()
            evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in evp:
                flush.zero_()
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize()
            pair[key] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evp) * 1e3
        wk = bwd_work(Bsz, Dm, L, N, in_bytes=2 if w.in_dtype == "bf16" else 4, dout_bytes=2)
        res[name] = {"batch": Bsz, "dim": Dm, "seqlen": L, "dstate": N, "dout_dtype": "bf16",
                     "us_per_call": secs * 1e6, "elems_per_s": wk["elements"] / secs,
                     "roofline": roofline_entry(wk, secs, sms, hbm_gbs, sm_mhz, rates=rates,
                                                traffic=recorded_traffic("selscan_bwd", name)),
                     "launches_per_call": launches, "gpu_launches": launches * reps,
                     "training_pair": dict(pair, note="selscan_fwd_ckpt keeps the state before every 16-step "
                                           "chunk; selscan_bwd_ckpt reruns chunks from it (no forward pass of "
                                           "its own)")}
        del t, g, ws, go, gh, out, ck
    return res


def run_decode(args, torch, ss, device, stream, flush, sms, hbm_gbs):
    """Secondary: the recurrent decode workload (64 steps of selscan_step carrying the fp32 state)."""
    w = si.WORKLOADS["decode_step"]
    inp = si.make_inputs(w)
    T = inp["steps"]
    Bsz, Dm, _, N = inp["shape"]
    t = {k: _dev(torch, inp.get(k), device) for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias", "h0")}
    state = t["h0"].clone()
    out = torch.empty((T, Bsz, Dm), device=device, dtype=torch.float32)

    def step(s):
        ss.selscan_step(t["u"][s], t["delta"][s], t["A"], t["B"][s], t["C"][s], state, D=t["D"], z=t["z"][s],
                        delta_bias=t["delta_bias"], out=out[s], stream=stream)

    for _ in range(2):
        state.copy_(t["h0"])
        for s in range(T):
            step(s)
    # Each step is timed on its own, after an L2 flush: the 84 MB state would otherwise stay partly
    # in the 126 MB L2 from one step to the next, which a model with many layers does not see.
    reps = 5
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(reps * T)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(reps * T)]
    for r in range(reps):
        state.copy_(t["h0"])
        for s in range(T):
            flush.zero_()
            starts[r * T + s].record(stream)
            step(s)
            ends[r * T + s].record(stream)
    torch.cuda.synchronize()
    per_rep = [sum(starts[r * T + s].elapsed_time(ends[r * T + s]) for s in range(T)) / 1e3 for r in range(reps)]
    secs = statistics.median(per_rep)
    wk = step_work(Bsz, Dm, N)
    gbs = wk["bytes"] * T / secs / 1e9
    return {"workload": "decode_step", "batch": Bsz, "dim": Dm, "dstate": N, "steps": T,
            "l2": "flushed (256 MiB write) before every step, outside its events",
            "elems_per_s": Bsz * Dm * T / secs, "us_per_step": secs / T * 1e6,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
                         "traffic": recorded_traffic("selscan_step", "decode_step")},
            "gpu_launches": T * reps}


# ------------------------------------------------------------------------------------------------
# CPU arms (the fp64 oracle)
# ------------------------------------------------------------------------------------------------

def _oracle_rate(inp, rows, nthreads):
    import oracle

    t0 = time.perf_counter()
    oracle.selscan_fwd(inp, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(inp, w, budget_cpu_s=15.0):
    """The fp64 oracle as it stands on all host cores, on a row sample sized for ~budget_cpu_s of CPU work."""
    Bsz, Dm, L, N = inp["shape"]
    cores = os.cpu_count() or 1
    probe_rows = list(range(min(8, Bsz * Dm)))
    per_row = _oracle_rate(inp, probe_rows, 1) / len(probe_rows)  # CPU seconds per row on one core
    nrows = int(max(cores, min(Bsz * Dm, budget_cpu_s / max(per_row, 1e-9))))
    nrows = min(nrows, Bsz * Dm)
    rng = np.random.default_rng(7)
    rows = sorted(rng.choice(Bsz * Dm, size=nrows, replace=False).tolist())
    secs = _oracle_rate(inp, rows, cores)
    return {"value": nrows * L / secs, "unit": "elems/s", "cores": cores, "kind": "oracle",
            "sample": f"{nrows} of {Bsz * Dm} (b,d) rows of {w.name}, each over its full L={L}, N={N}",
            "seconds": secs}


def run_reference(args):
    """The oracle arm: each step runs the fp64 oracle on a bounded row sample of the workload."""
    w = si.WORKLOADS[args.workload]
    inp = si.make_inputs(w)
    Bsz, Dm, L, N = inp["shape"]
    cores = os.cpu_count() or 1
    per_row = _oracle_rate(inp, list(range(min(8, Bsz * Dm))), 1) / min(8, Bsz * Dm)
    total_steps = args.steps + args.warmup
    budget_wall = 150.0 / max(total_steps, 1)  # the whole run stays within a few minutes
    nrows = int(min(Bsz * Dm, max(1, budget_wall * cores / max(per_row, 1e-9))))
    rng = np.random.default_rng(11)
    rows = sorted(rng.choice(Bsz * Dm, size=nrows, replace=False).tolist())
    for _ in range(args.warmup):
        _oracle_rate(inp, rows, cores)
    times = [_oracle_rate(inp, rows, cores) for _ in range(args.steps)]
    secs = sum(times)
    value = nrows * L * args.steps / secs
    sample = f"{nrows} of {Bsz * Dm} (b,d) rows of {w.name} per step, each over its full L={L}, N={N}"
    return {"metric": METRIC, "value": value, "unit": "elems/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(w, Bsz, L),
            "cpu_baseline": {"value": value, "unit": "elems/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "elems/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=[n for n in si.WORKLOAD_ORDER
                                                                     if not si.WORKLOADS[n].steps])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="CPU-seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-options", action="store_true", help="skip the reverse / zero-order-hold timings")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward (selscan_bwd) timings")
    ap.add_argument("--no-sweep", action="store_true", help="skip the other forward workloads")
    ap.add_argument("--sweep-steps", type=int, default=50)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist_mod

        torch.cuda.set_device(local_rank)
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = dist_mod
    res = run_ours(args, rank, world, local_rank, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
