#!/usr/bin/env python
"""Selective-scan bench: scanned elements per second (Bsz*Dch*L) of one
training-and-decode pass of the whole hot path on one workload.

One step = ss_scan_fwd (discretise, scan, contract, skip, gate) +
ss_scan_bwd (its three stages: segment states, reverse pass, reduction) +
one ss_step decode token continuing from the forward's final state (+ for
N > 1 the all-reduce of dA, dD, ddelta_bias across replicas).

Workload: the Mamba-130M-shaped layer Bsz=8, Dch=1536, L=2048, N=16 with bf16
inputs/outputs and float32 state and accumulation; synthetic seeded data
(u, z, B, C, delta_raw, dy ~ N(0,1); A[d,n] = -(n+1); D ~ N(0,1); delta_bias
= inverse softplus of dt, dt log-uniform in [1e-3, 1e-1]).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle (the method as plain sequential code) on a bounded sample of the same
workload on this machine's host cores.

Besides the step, rank 0 adds side measurements to the line (each with its
roofline): the decode step at Bsz=256, Dch=5120; conv1d + silu forward and
backward; the tensor-core input projection (x_proj + dt_proj); the fp32
Mamba-370M layer forward + backward; the long-sequence forward
(1 x 5120 x 131072); the bench layer with 64 states; and a four-piece chunked
prefill continued from the carried state.  ``--profile-workload`` runs only
one workload's kernels, for an ncu capture.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "selective-scan Gelem/s (B·D·L), fwd and fwd+bwd; % of HBM/MUFU roofline"
UNIT = "Gelem/s"
CFG_INDEX = 1
N_STATE = 16

# Hardware figures for the roofline denominators (one B300).
SMS = 148
SM_MAX_MHZ = 2032.0
FP32_LANES = 128            # FP32 operations per clock per SM
MUFU_LANES = 32             # MUFU (ex2 / lg2 / rcp) results per clock per SM, measured
FP32_PEAK_T = SMS * FP32_LANES * SM_MAX_MHZ * 1e6 / 1e12   # 38.49 T ops/s
MUFU_PEAK_T = SMS * MUFU_LANES * SM_MAX_MHZ * 1e6 / 1e12   # 9.62 T ops/s
L2_BYTES = 126 * 2 ** 20
# kernels one step launches: forward 1; backward states 2 (chunk summaries,
# chunk carries), reverse 1, reduce 2 (dB/dC, dA/dD/dbias); decode step 1
LAUNCHES_PER_STEP = 7


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# ---------------------------------------------------------------------------
# Algorithmic work per scanned element (b, d, t) of each stage, N = 16,
# s = bytes per I/O element, Dch = channels: what the method needs, not what
# a kernel executes.  fp32 = FP32 add/mul/fma operations, mufu = exp / log /
# reciprocal evaluations, bytes = each tensor read or written once.
#   fwd:          per state: delta*A, delta*u*B, the state update, C*h (4N);
#                 softplus 4, D skip 1, delta*u 1, gate 3; MUFU: N decays,
#                 softplus 2, sigmoid 2.  Bytes: u, delta, z in, y out (4s)
#                 plus B, C once per (b, t): 2Ns/Dch.
#   bwd_states:   chunk summaries: per state delta*A, the input term, the
#                 state fold, the decay product, yhat*C, the adjoint fold
#                 (6N) + 12; MUFU N + 4.  Bytes: u, delta, z, dy in (4s) +
#                 B, C + 33 floats out per 128 steps.
#   bwd_reverse:  the backward proper: per state the recomputed decay and
#                 state (3), adjoint (2), dC, dB, du-sum, ddelta-sum (2),
#                 dA, pre-gate output (7) = 12N; + 20 per element; MUFU N + 6.
#                 Bytes: u, delta, z, dy in, du, ddelta, dz out (7s), B, C,
#                 dB, dC written once per (b, t): (2Ns + 8N)/Dch.
#   bwd_reduce:   dB/dC partials of 128-row blocks read, dB, dC written:
#                 2N*4*(ceil(Dch/128) + 1)/Dch.
# ---------------------------------------------------------------------------
def kernel_work(s, Dch, N=N_STATE):
    G = (Dch + 127) // 128
    return {
        "fwd": dict(fp32=4 * N + 9, mufu=N + 4, bytes=4 * s + 2 * N * s / Dch),
        "bwd_states": dict(fp32=6 * N + 12, mufu=N + 4,
                           bytes=4 * s + 2 * N * s / Dch + 33 * 4 / 128),
        "bwd_reverse": dict(fp32=12 * N + 20, mufu=N + 6,
                            bytes=7 * s + (2 * N * s + 8 * N) / Dch),
        "bwd_reduce": dict(fp32=0, mufu=0, bytes=2 * N * 4 * (G + 1) / Dch),
    }


def roofline(name, work, elems, ms, hbm_gbs, traffic=None):
    """Roofline of one kernel: the binding resource is the one whose
    algorithmic work takes longest at its peak; achieved = that work / the
    measured time."""
    t = ms * 1e-3
    times = {"hbm": work["bytes"] * elems / (hbm_gbs * 1e9),
             "fp32": work["fp32"] * elems / (FP32_PEAK_T * 1e12),
             "mufu": work["mufu"] * elems / (MUFU_PEAK_T * 1e12)}
    res = max(times, key=times.get)
    base = {"kernel": name, "traffic": traffic, "resource": res,
            "algorithmic_bytes": work["bytes"] * elems, "algorithmic_fp32": work["fp32"] * elems,
            "algorithmic_mufu": work["mufu"] * elems,
            "bound_ms": {k: round(v * 1e3, 4) for k, v in times.items()}}
    if res == "hbm":
        ach = work["bytes"] * elems / t / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(ach / hbm_gbs, 4), **base}
    peak = FP32_PEAK_T if res == "fp32" else MUFU_PEAK_T
    ach = work[res] * elems / t / 1e12
    return {"bound": "alu", "achieved": round(ach, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
            "frac": round(ach / peak, 4), **base}


# The sources the step's kernels (forward, backward, decode token) are built
# from: ncu traffic taken on other versions of these files is not reported.
STEP_SOURCES = ("common.cuh", "launch.h", "scan_fwd.cu", "scan_bwd.cu", "step.cu")


def csrc_digest():
    h = hashlib.sha256()
    for name in STEP_SOURCES:
        h.update(open(os.path.join(ROOT, "selective_state_space_114_b300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, when it was
    taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("csrc_digest") != csrc_digest():
        return None
    v = d.get("kernels", {}).get(kernel)
    return None if v is None else v.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs:
    NVML when its library loads, else ``nvidia-smi --query-gpu ... -lms``."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index=0):
        self.samples = []   # (sm_mhz, reasons bitmask or list of names)
        self._stop = threading.Event()
        self.mode = None
        self.max_mhz = None
        self.err = []
        self.bus = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            self.bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id,
                                             props.pci_device_id)
        except Exception as e:
            self.err.append(f"pci id: {e}")
        try:
            import pynvml as nv
            nv.nvmlInit()
            self.nv = nv
            self.h = (nv.nvmlDeviceGetHandleByPciBusId(self.bus.encode()) if self.bus
                      else nv.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(self.h, nv.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:
            self.err.append(f"nvml: {e}")
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "nvidia-smi"

    def _nvml_reasons(self):
        nv = self.nv
        try:
            return nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        except Exception:
            return nv.nvmlDeviceGetCurrentClocksThrottleReasons(self.h)

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                     int(self._nvml_reasons())))
            except Exception:
                pass
            time.sleep(0.002)

    def _start_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "20"]
        if self.bus:
            cmd += ["-i", self.bus]
        self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                      text=True)
        time.sleep(0.3)  # let it take its first samples before the timed region

    def _stop_smi(self):
        self._proc.terminate()
        out, _ = self._proc.communicate(timeout=10)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                mhz, mx = float(f[0]), float(f[1])
                active = int(f[2], 16) if f[2].startswith("0x") else 0
            except ValueError:
                continue
            self.max_mhz = mx
            seen = [nm for nm, v in zip(names, f[3:7]) if v.lower() == "active"]
            self.samples.append((mhz, active, seen))

    def __enter__(self):
        if self.mode == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        elif self.mode == "nvidia-smi":
            try:
                self._start_smi()
            except Exception as e:
                self.err.append(f"nvidia-smi: {e}")
                self.mode = None
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self._t.join()
        elif self.mode == "nvidia-smi":
            try:
                self._stop_smi()
            except Exception as e:
                self.err.append(f"nvidia-smi: {e}")

    def summary(self):
        if not self.mode:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks not sampled"],
                    "errors": self.err}
        busy = [s for s in self.samples if not (s[1] & 0x1)] or self.samples
        seen = set()
        for s in busy:
            for bit, nm in self.REASONS.items():
                if s[1] & bit:
                    seen.add(nm)
            if len(s) > 2:
                seen.update(s[2])
        mhz = statistics.median([s[0] for s in busy]) if busy else None
        return {"sm_mhz": mhz, "sm_max_mhz": self.max_mhz, "reasons": sorted(seen),
                "samples": len(busy), "source": self.mode}


# ---------------------------------------------------------------------------
# distributed set-up
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def workload_config(world):
    cfg = synth.config(CFG_INDEX)
    E = cfg["Bsz"] * cfg["Dch"] * cfg["L"]
    per_step_mb = (8 * E * 2 + 8 * E * 2) / 2 ** 20
    return cfg, {
        "workload": "mamba130m-shaped selective-scan layer: Bsz=8 Dch=1536 L=2048 N=16, bf16 "
                    "I/O, f32 state; step = fwd + bwd (3 stages) + 1 decode token",
        "Bsz": cfg["Bsz"], "Dch": cfg["Dch"], "L": cfg["L"], "N": cfg["N"], "io_dtype": "bf16",
        "softplus": True, "gate": True, "global_batch": cfg["Bsz"] * world,
        "parallelism": "replicas" if world == 1 else f"dp{world} (param-grad all-reduce)",
        "l2": f"inputs larger than L2: ~{per_step_mb:.0f} MiB of activations and gradients "
              f"touched per step vs {L2_BYTES // 2**20} MiB L2; no flush",
    }


# ---------------------------------------------------------------------------
# CPU (oracle) timing
# ---------------------------------------------------------------------------
def oracle_sample_step(cfg, nch, seed):
    """One fp64 oracle pass (fwd + bwd + one step) over all Bsz batches of
    the first ``nch`` channels, L = full length.  Returns seconds."""
    import oracle
    sub = dict(cfg, Dch=nch)
    x = synth.make_inputs(sub, seed=seed, with_dy=True)
    w = {k: synth.widen(v) for k, v in x.items()}
    t0 = time.perf_counter()
    _, h = oracle.scan_fwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                           w["delta_bias"], True)
    oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                    w["delta_bias"], True, w["dy"])
    tok = synth.step_inputs(dict(sub, L=1), 0, seed=seed)
    tw = {k: synth.widen(v) for k, v in tok.items()}
    oracle.step(h, tw["u"], tw["delta"], w["A"], tw["B"], tw["C"], w["D"], tw["z"],
                w["delta_bias"], True)
    return time.perf_counter() - t0


def size_oracle_sample(cfg, target_s, seed):
    """Number of channels (all batches, full L) whose oracle pass takes about
    target_s seconds on the host cores (capped at the whole workload)."""
    cores = os.cpu_count() or 1
    n = max(2, min(cores, 8))
    for _ in range(4):
        t = oracle_sample_step(cfg, n, seed)
        if t >= 0.5 * target_s or n >= cfg["Dch"]:
            break
        n = int(min(cfg["Dch"], max(2 * n, n * target_s / max(t, 1e-6))))
    return n


def cpu_baseline(cfg, seed, target_s=12.0):
    """The oracle as it stands, timed on the host cores: passes over the
    first n channels (all batches, full L), repeated while the sample is
    shorter than about target_s seconds."""
    import oracle
    cores = oracle.default_threads()
    n = size_oracle_sample(cfg, target_s, seed)
    t = oracle_sample_step(cfg, n, seed)
    reps = 1
    while t < 0.5 * target_s and reps < 64:
        t += oracle_sample_step(cfg, n, seed)
        reps += 1
    elems = cfg["Bsz"] * n * cfg["L"] * reps
    return {"value": round(elems / t / 1e9, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} fp64 oracle pass(es) of fwd+bwd+1 step over all {cfg['Bsz']} "
                      f"batches x first {n} of {cfg['Dch']} channels x L={cfg['L']} "
                      f"({elems} elements, {t:.1f} s)"}


def run_reference(args):
    world, rank, _ = dist_env()
    cfg, conf = workload_config(1)
    if rank != 0:
        return 0
    import oracle
    cores = oracle.default_threads()
    W, K = max(3, args.warmup), args.steps
    budget = 150.0  # seconds for the whole run
    per_step = max(0.5, budget / (W + K))
    n = size_oracle_sample(cfg, per_step, cfg["seed"])
    for _ in range(W):
        oracle_sample_step(cfg, n, cfg["seed"])
    times = [oracle_sample_step(cfg, n, cfg["seed"]) for _ in range(K)]
    elems = cfg["Bsz"] * n * cfg["L"]
    ms = 1e3 * sum(times) / K
    value = elems / (ms * 1e-3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": conf,
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 oracle fwd+bwd+1 decode step over all "
                                   f"{cfg['Bsz']} batches x first {n} of {cfg['Dch']} channels x "
                                   f"L={cfg['L']} ({elems} elements)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------
def _flushed_median_ms(fn, steps, dev):
    """Median time of fn() with L2 flushed before each call (a 256 MiB read).
    The GPU first spins for ~25 ms so that the host enqueues every timed call
    ahead of it: the events then bracket GPU work only, not launch latency."""
    import torch
    flush = torch.ones(64 * 2 ** 20, device=dev, dtype=torch.float32)
    sink = torch.empty((), device=dev, dtype=torch.float32)
    for _ in range(3):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)
    for e0, e1 in evs:
        torch.sum(flush, dim=0, out=sink)
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def conv_measure(ss, dev, seed, steps=16):
    """The causal depthwise conv1d + silu (width 4) that produces u, forward
    and backward, on the bench layer's shape (8 x 1536 x 2048, bf16); L2 is
    flushed before each call.  Returns times and HBM rooflines."""
    import torch
    cfg = synth.config(CFG_INDEX)
    Bsz, Dch, L, K = cfg["Bsz"], cfg["Dch"], cfg["L"], 4
    E = Bsz * Dch * L
    bf = torch.bfloat16
    x = torch.from_numpy(synth.normal(seed, 20, E, "bf16").reshape(Bsz, Dch, L)).view(bf).to(dev)
    g = torch.from_numpy(synth.normal(seed, 23, E, "bf16").reshape(Bsz, Dch, L)).view(bf).to(dev)
    w = torch.from_numpy(synth.normal(seed, 21, Dch * K, "f32").reshape(Dch, K) / 2.0).to(dev)
    b = torch.from_numpy(synth.normal(seed, 22, Dch, "f32")).to(dev)
    u = torch.empty_like(x)
    grads = {"dx": torch.empty_like(x), "dw": torch.empty((Dch, K), device=dev),
             "dbias": torch.empty((Dch,), device=dev)}
    ms_f = _flushed_median_ms(lambda: ss.ss_conv1d_silu(x, w, b, True, out=u), steps, dev)
    ms_b = _flushed_median_ms(lambda: ss.ss_conv1d_silu_bwd(x, w, b, True, g, out=grads), steps,
                              dev)
    hbm, _ = load_peaks()
    res = {"workload": f"conv1d (width {K}) + silu, Bsz={Bsz} Dch={Dch} L={L}, bf16, "
                       f"L2 flushed before each call"}
    for name, ms, nbytes in (("fwd", ms_f, 2 * 2 * E), ("bwd", ms_b, 3 * 2 * E)):
        ach = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "gelem_s": round(E / (ms * 1e-3) / 1e9, 2), "bound": "hbm",
                     "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(ach / hbm, 4), "algorithmic_bytes": nbytes}
    return res
def xproj_measure(ss, dev, seed, steps=16):
    """The input projection (x_proj then dt_proj on the tensor cores) on the
    bench layer's shape (8 x 1536 x 2048, dt_rank 48, N = 16, bf16), L2
    flushed before each call.  HBM-bound: u read, delta, B, C written."""
    import torch
    cfg = synth.config(CFG_INDEX)
    Bsz, Dch, L, N, R = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"], 48
    E = Bsz * Dch * L
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    bf = torch.bfloat16
    u = torch.randn((Bsz, Dch, L), generator=gen, device=dev).to(bf)
    Wx = (torch.randn((R + 2 * N, Dch), generator=gen, device=dev) / Dch ** 0.5).to(bf)
    Wdt = (torch.randn((Dch, R), generator=gen, device=dev) / R ** 0.5).to(bf)
    out = (torch.empty_like(u), torch.empty((Bsz, N, L), device=dev, dtype=bf),
           torch.empty((Bsz, N, L), device=dev, dtype=bf))
    ms = _flushed_median_ms(lambda: ss.ss_xproj(u, Wx, Wdt, N, out=out), steps, dev)
    nbytes = 2 * E * 2 + 2 * 2 * Bsz * N * L + 2 * (R + 2 * N) * Dch + 2 * Dch * R
    flops = 2 * Bsz * L * Dch * (R + 2 * N) + 2 * Bsz * L * R * Dch
    hbm, _ = load_peaks()
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"x_proj + dt_proj, Bsz={Bsz} Dch={Dch} L={L} dt_rank={R} N={N}, bf16, "
                        f"L2 flushed before each call",
            "ms": round(ms, 4), "bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(ach / hbm, 4), "algorithmic_bytes": nbytes,
            "tensor_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "wait_failures": ss.ss_xproj_wait_failures()}


def decode_step_measure(ss, dev, seed, steps=16):
    """The one-token step on the decode workload (Bsz=256, Dch=5120, N=16,
    bf16 tokens, float32 state): its state (84 MB) fits in L2, so L2 is
    flushed before each timed step by reading a 256 MiB buffer (a read leaves
    no dirty lines to be written back during the step); the events bracket
    the step kernel only.  Returns its time and HBM roofline."""
    import torch
    cfg = synth.config(4)
    Bsz, Dch, N = cfg["Bsz"], cfg["Dch"], cfg["N"]
    x = synth.make_inputs(dict(cfg, L=1), seed=seed)
    tok = synth.step_inputs(cfg, 0, seed=seed)
    bf = torch.bfloat16

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).view(bf).to(dev)

    u, dl, z, B, C = (t(tok[k]) for k in ("u", "delta", "z", "B", "C"))
    A = torch.from_numpy(np.ascontiguousarray(x["A"], dtype=np.float32)).to(dev)
    D = torch.from_numpy(np.ascontiguousarray(x["D"], dtype=np.float32)).to(dev)
    bias = torch.from_numpy(np.ascontiguousarray(x["delta_bias"], dtype=np.float32)).to(dev)
    h = torch.zeros((Bsz, Dch, N), device=dev, dtype=torch.float32)
    y = torch.empty((Bsz, Dch), device=dev, dtype=bf)
    ms = _flushed_median_ms(lambda: ss.ss_step(h, u, dl, A, B, C, D, z, bias, True, out=y), steps,
                            dev)
    rows = Bsz * Dch
    nbytes = rows * (2 * N * 4 + 4 * 2) + 2 * Bsz * N * 2  # h in/out, u/delta/z/y, B/C
    hbm, _ = load_peaks()
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"decode step Bsz={Bsz} Dch={Dch} N={N}, bf16 tokens, f32 state, "
                        f"L2 flushed before each step", "ms": round(ms, 4),
            "bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(ach / hbm, 4), "algorithmic_bytes": nbytes}


def _device_inputs(cfg, dev, seed, with_dy=False):
    """Inputs of a workload made on the device: activations and B/C drawn from
    N(0, 1) by torch's seeded generator (the workload's distributions, not the
    host generator's values; timing does not depend on them), A, D and
    delta_bias from the host generator."""
    import torch
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    dtype = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def rnd(*shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(dtype)

    x = {"u": rnd(Bsz, Dch, L), "delta": rnd(Bsz, Dch, L), "z": rnd(Bsz, Dch, L),
         "B": rnd(Bsz, N, L), "C": rnd(Bsz, N, L)}
    if with_dy:
        x["dy"] = rnd(Bsz, Dch, L)
    x["A"] = torch.from_numpy(synth.param_A(Dch, N)).to(dev)
    x["D"] = torch.from_numpy(synth.param_D(seed, Dch)).to(dev)
    x["delta_bias"] = torch.from_numpy(synth.param_delta_bias(seed, Dch, cfg["dt_range"])).to(dev)
    return x, dtype


def _timed_ms(fns, steps, dev):
    """Mean device time of each function in fns over `steps` back-to-back
    rounds (inputs far larger than L2, so no flush), after 3 warm-up rounds."""
    import torch
    for _ in range(3):
        for f in fns:
            f()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)
    for row in evs:
        row[0].record()
        for i, f in enumerate(fns):
            f()
            row[i + 1].record()
    torch.cuda.synchronize()
    return [statistics.mean(r[i].elapsed_time(r[i + 1]) for r in evs) for i in range(len(fns))]


def configs_measure(ss, dev, seed):
    """The other full-size workloads: the fp32 Mamba-370M-shaped layer forward
    and backward (8 x 2048 x 2048) and the long-sequence bf16 forward
    (1 x 5120 x 131072), each kernel stage with its roofline."""
    import torch
    hbm, _ = load_peaks()
    out = {}
    cfg = synth.config(2)
    x, dtype = _device_inputs(cfg, dev, seed + 2, with_dy=True)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    y = torch.empty_like(x["u"])
    g = {"du": torch.empty_like(y), "ddelta": torch.empty_like(y), "dz": torch.empty_like(y),
         "dA": torch.empty((Dch, N), device=dev), "dB": torch.empty((Bsz, N, L), device=dev),
         "dC": torch.empty((Bsz, N, L), device=dev), "dD": torch.empty((Dch,), device=dev),
         "ddelta_bias": torch.empty((Dch,), device=dev)}
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_F32), device=dev,
                     dtype=torch.uint8)
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    fns = [lambda: ss.ss_scan_fwd(*args, out=y)]
    names = ["fwd", "bwd_states", "bwd_reverse", "bwd_reduce"]
    for st in ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce"):
        fns.append(lambda st=st: ss.ss_scan_bwd(*args, x["dy"], workspace=ws, out=g,
                                                stages=(st,)))
    ms = _timed_ms(fns, 10, dev)
    work = kernel_work(4, Dch)
    tot = sum(ms)
    out["mamba370m_fp32_fwd_bwd"] = {
        "workload": f"Bsz={Bsz} Dch={Dch} L={L} N={N}, fp32 I/O, fwd + bwd, inputs larger than L2",
        "gelem_s": round(E / (tot * 1e-3) / 1e9, 3), "ms": round(tot, 4),
        "kernels": {nm: {"ms": round(t, 4), **{k: v for k, v in roofline(nm, work[nm], E, t, hbm)
                                               .items() if k in ("bound", "achieved", "peak",
                                                                 "unit", "frac", "resource")}}
                    for nm, t in zip(names, ms)}}
    del x, y, g, ws
    torch.cuda.empty_cache()

    cfg = synth.config(3)
    x, dtype = _device_inputs(cfg, dev, seed + 3)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    y = torch.empty_like(x["u"])
    h = torch.empty((Bsz, Dch, N), device=dev)
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    (t,) = _timed_ms([lambda: ss.ss_scan_fwd(*args, out=y, h_last=h, return_last_state=True)],
                     5, dev)
    r = roofline("fwd", kernel_work(2, Dch)["fwd"], E, t, hbm)
    out["long_sequence_bf16_fwd"] = {
        "workload": f"Bsz={Bsz} Dch={Dch} L={L} N={N}, bf16 I/O, f32 state, fwd, "
                    f"inputs larger than L2",
        "gelem_s": round(E / (t * 1e-3) / 1e9, 3), "ms": round(t, 4),
        **{k: v for k, v in r.items() if k in ("bound", "achieved", "peak", "unit", "frac",
                                               "resource")}}
    del x, y, h
    torch.cuda.empty_cache()

    # the bench layer (8 x 1536 x 2048, bf16) with 64 states, forward and backward
    cfg = dict(synth.config(1), N=64)
    x, dtype = _device_inputs(cfg, dev, seed + 5, with_dy=True)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    y = torch.empty_like(x["u"])
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_BF16), device=dev,
                     dtype=torch.uint8)
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    g = ss.ss_scan_bwd(*args, x["dy"], workspace=ws)
    fns = [lambda: ss.ss_scan_fwd(*args, out=y)]
    for st in ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce"):
        fns.append(lambda st=st: ss.ss_scan_bwd(*args, x["dy"], workspace=ws, out=g,
                                                stages=(st,)))
    ms = _timed_ms(fns, 5, dev)
    work = kernel_work(2, Dch, N)
    out["state_size_64_bf16_fwd_bwd"] = {
        "workload": f"Bsz={Bsz} Dch={Dch} L={L} N={N}, bf16 I/O, fwd + bwd, inputs larger than L2",
        "gelem_s": round(E / (sum(ms) * 1e-3) / 1e9, 3), "ms": round(sum(ms), 4),
        "kernels": {nm: {"ms": round(t, 4), **{k: v for k, v in roofline(nm, work[nm], E, t, hbm)
                                               .items() if k in ("bound", "achieved", "peak",
                                                                 "unit", "frac", "resource")}}
                    for nm, t in zip(["fwd", "bwd_states", "bwd_reverse", "bwd_reduce"], ms)}}
    del x, y, g, ws
    torch.cuda.empty_cache()

    # chunked prefill: the bench layer's forward as four 512-step pieces, each
    # continuing from the state the previous one left (updated in place)
    cfg = synth.config(1)
    x, dtype = _device_inputs(cfg, dev, seed + 6)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    P = 4
    Lp = L // P
    pieces = [{k: x[k][..., i * Lp:(i + 1) * Lp].contiguous() for k in ("u", "delta", "z", "B",
                                                                       "C")}
              for i in range(P)]
    ys = [torch.empty_like(pc["u"]) for pc in pieces]
    h = torch.zeros((Bsz, Dch, N), device=dev)

    def prefill():
        for i, pc in enumerate(pieces):
            ss.ss_scan_fwd(pc["u"], pc["delta"], x["A"], pc["B"], pc["C"], x["D"], pc["z"],
                           x["delta_bias"], True, out=ys[i], return_last_state=True,
                           h0=h if i else None, h_last=h)

    (t,) = _timed_ms([prefill], 10, dev)
    r = roofline("fwd", kernel_work(2, Dch)["fwd"], E, t, hbm)
    out["chunked_prefill_bf16_fwd"] = {
        "workload": f"Bsz={Bsz} Dch={Dch} L={L} N={N} as {P} pieces of {Lp} steps continued "
                    f"from the carried state (ss_scan_fwd_from_state), bf16 I/O",
        "gelem_s": round(E / (t * 1e-3) / 1e9, 3), "ms": round(t, 4),
        **{k: v for k, v in r.items() if k in ("bound", "achieved", "peak", "unit", "frac",
                                               "resource")}}
    del x, pieces, ys, h
    torch.cuda.empty_cache()
    return out


def run_profile_workload(args):
    """Run a workload's kernels `--profile-iters` times and exit, for an ncu
    capture of one launch: mamba370m (the fp32 8 x 2048 x 2048 layer, forward
    then backward) or long_sequence (the bf16 1 x 5120 x 131072 forward; the
    length may be cut with --profile-L to keep a capture small)."""
    import torch
    import selective_state_space_114_b300 as ss
    dev = torch.device("cuda", 0)
    ci = {"mamba370m": 2, "long_sequence": 3}[args.profile_workload]
    cfg = synth.config(ci)
    if args.profile_L:
        cfg = dict(cfg, L=args.profile_L)
    x, _ = _device_inputs(cfg, dev, cfg["seed"], with_dy=(ci == 2))
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    args_ = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y = torch.empty_like(x["u"])
    ws = None
    if ci == 2:
        ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_F32), device=dev,
                         dtype=torch.uint8)
    for _ in range(args.profile_iters):
        ss.ss_scan_fwd(*args_, out=y)
        if ws is not None:
            ss.ss_scan_bwd(*args_, x["dy"], workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_workload": args.profile_workload, "Bsz": Bsz, "Dch": Dch, "L": L,
                      "iters": args.profile_iters}))
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if args.gpus != world:
        if world == 1 and args.gpus > 1:
            raise SystemExit("bench.py --gpus N>1 must be launched with torch.distributed.run")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import selective_state_space_114_b300 as ss
    from selective_state_space_114_b300 import dist as sdist

    dev = torch.device("cuda", local)
    cfg, conf = workload_config(world)
    seed = sdist.rank_seed(cfg["seed"], rank)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    W, K = max(3, args.warmup), args.steps

    x = synth.make_inputs(cfg, seed=seed, with_dy=True)
    tok = synth.step_inputs(dict(cfg, L=1), 0, seed=seed)

    def host(a, pin=True):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.pin_memory() if pin else t

    hx = {k: host(v) for k, v in x.items()}
    ht = {k: host(v) for k, v in tok.items()}
    d = {k: v.to(dev) for k, v in hx.items()}
    dt = {k: v.to(dev) for k, v in ht.items()}
    bf = torch.bfloat16
    y = torch.empty((Bsz, Dch, L), device=dev, dtype=bf)
    h = torch.empty((Bsz, Dch, N), device=dev, dtype=torch.float32)
    g = {"du": torch.empty_like(y), "ddelta": torch.empty_like(y), "dz": torch.empty_like(y),
         "dA": torch.empty((Dch, N), device=dev), "dB": torch.empty((Bsz, N, L), device=dev),
         "dC": torch.empty((Bsz, N, L), device=dev), "dD": torch.empty((Dch,), device=dev),
         "ddelta_bias": torch.empty((Dch,), device=dev)}
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_BF16), device=dev,
                     dtype=torch.uint8)
    yt = torch.empty((Bsz, Dch), device=dev, dtype=bf)
    stages = ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce")
    names = ["fwd", "bwd_states", "bwd_reverse", "bwd_reduce", "step"]

    def one_step(evs=None, src=None):
        if src is not None:  # e2e: this step's inputs arrive from pinned host memory
            for k, v in src[0].items():
                d[k].copy_(v, non_blocking=True)
            for k, v in src[1].items():
                dt[k].copy_(v, non_blocking=True)
        rec = (lambda i: evs[i].record()) if evs is not None else (lambda i: None)
        rec(0)
        ss.ss_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                       d["delta_bias"], True, return_last_state=True, out=y, h_last=h)
        rec(1)
        for i, st in enumerate(stages):
            ss.ss_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                           d["delta_bias"], True, d["dy"], workspace=ws, out=g, stages=(st,))
            rec(2 + i)
        ss.ss_step(h, dt["u"], dt["delta"], d["A"], dt["B"], dt["C"], d["D"], dt["z"],
                   d["delta_bias"], True, out=yt)
        rec(5)
        if world > 1:
            sdist.allreduce_param_grads(g)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(W):
        one_step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record()
        for k in range(K):
            one_step(evs[k])
        end.record()
        torch.cuda.synchronize()
    barrier()
    ms_local = start.elapsed_time(end) / K
    ms = sdist.max_over_ranks(ms_local, device=dev)
    per_kernel = {nm: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K))
                  for i, nm in enumerate(names)}
    value = world * E / (ms * 1e-3) / 1e9
    fwd_gelem = E / (per_kernel["fwd"] * 1e-3) / 1e9

    decode = decode_step_measure(ss, dev, seed) if rank == 0 else None
    conv = conv_measure(ss, dev, seed) if rank == 0 else None
    others = configs_measure(ss, dev, seed) if rank == 0 else None
    xproj = xproj_measure(ss, dev, seed) if rank == 0 else None

    # end to end through the public API with host buffers
    Ke = max(3, min(K, 10))
    outs = {"y": y, "yt": yt, **g}
    hout = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(v.numel() * v.element_size() for v in list(hx.values()) + list(ht.values()))
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(Ke):
        one_step(src=(hx, ht))
        for k, v in outs.items():
            hout[k].copy_(v, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    barrier()
    e2e_ms = sdist.max_over_ranks(e0.elapsed_time(e1) / Ke, device=dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm, peak_src = load_peaks()
    work = kernel_work(2, Dch)
    roofs = {nm: roofline(nm, work[nm], E, per_kernel[nm], hbm, ncu_traffic(nm))
             for nm in names if nm in work}
    dominant = max(roofs, key=lambda nm: per_kernel[nm])
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": conf,
        "fwd_gelem_s": round(fwd_gelem, 3),
        "roofline": roofs[dominant],
        "roofline_peak_source": f"fp32: {SMS} SMs x {FP32_LANES} ops/clk x {SM_MAX_MHZ} MHz; "
                                f"mufu: {SMS} SMs x {MUFU_LANES} ops/clk (measured) x "
                                f"{SM_MAX_MHZ} MHz; hbm: {hbm} GB/s of {peak_src}",
        "kernels": {nm: {"ms": round(per_kernel[nm], 4),
                         "share": round(per_kernel[nm] / sum(per_kernel.values()), 4),
                         **({"frac": roofs[nm]["frac"], "bound": roofs[nm]["bound"]}
                            if nm in roofs else {})} for nm in names},
        "gpu_launches": K * LAUNCHES_PER_STEP,
        "decode_step": decode,
        "conv1d_silu": conv,
        "other_workloads": others,
        "xproj": xproj,
        "e2e": {"value": round(world * E / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 3)},
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, seed)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing on the host cores")
    ap.add_argument("--profile-workload", choices=["mamba370m", "long_sequence"],
                    help="only run that workload's kernels (for an ncu capture) and exit")
    ap.add_argument("--profile-L", type=int, default=0)
    ap.add_argument("--profile-iters", type=int, default=2)
    args = ap.parse_args()
    if args.profile_workload:
        return run_profile_workload(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
