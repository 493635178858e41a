#!/usr/bin/env python
"""Selective-scan bench: scanned elements per second (B*D*L) of the whole hot
path, with the roofline of every kernel and the fp64 oracle timed beside it.

Headline step (the JSON line's ``value``): one pass of the whole path over the
Mamba-130M-shaped layer (Bsz=8, Dch=1536, L=2048, N=16, bf16 I/O, float32
state): the forward, keeping the chunk states for the backward
(ss_scan_fwd_save) + its backward (ss_scan_bwd_saved's three stages) + one
ss_step decode token continuing from the forward's final state (+ for N > 1
replicas the all-reduce of dA, dD, ddelta_bias).  The backward that
recomputes the chunk states (ss_scan_bwd) is timed beside it.  Synthetic seeded data with the
workload's distributions (u, z, B, C, delta_raw, dy ~ N(0,1); A[d,n] =
-(n+1); D ~ N(0,1); delta_bias = inverse softplus of dt, dt log-uniform in
[1e-3, 1e-1]).

``configs`` in the line: each workload of the pages' configuration list with
its own time, Gelem/s, roofline and fp64 oracle sample on the host cores --
the Mamba-130M layer forward, the fp32 Mamba-370M layer forward + backward,
the long-sequence forward (1 x 5120 x 131072) and the decode workload (128
successive steps, 256 x 5120, state updated in place).

Roofline counts follow the method, per scanned element (b, d, t), N states,
s bytes per I/O element: forward 4N+10 FP32 operations and N+4 MUFU
evaluations, backward 10N+10 and N+6 (the whole backward: the chunk
summaries the kernels run first are part of its time, not extra work),
bytes = each tensor read or written once.  The FP32 and MUFU peaks are per-SM
rates measured by the microbenchmark built beside the library
(``selective_state_space_114_b300/probe/pipes.cu``) times the SM count and
the maximum SM clock; HBM is the measured copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--no-cpu-baseline] [--pipes] [--profile-workload NAME]

``--impl reference`` times the fp64 CPU oracle (the method as plain
sequential code) on a bounded sample of the headline workload.  ``--pipes``
prints the microbenchmark's rates and exits.  ``--profile-workload`` runs one
workload's kernels a few times and exits, for an ncu capture.
"""
from __future__ import annotations

import argparse
import ctypes
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
SMS = 148
SM_MAX_MHZ = 2032.0
L2_BYTES = 126 * 2 ** 20
# kernels one headline step launches: forward 1; backward summaries 2 (chunk
# summaries, chunk carries), reverse 1, reductions 2 (dB/dC, dA/dD/dbias);
# decode step 1
LAUNCHES_PER_STEP = 7
# per-SM rates used when the microbenchmark cannot run (its last results on
# this pool): FP32 operations, MUFU ex2 evaluations per SM clock
FALLBACK_PIPES = {"ffma": 124.3, "ex2": 31.98}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# ---------------------------------------------------------------------------
# pipe rates (microbenchmark) and peaks
# ---------------------------------------------------------------------------
PIPE_TESTS = {"ex2": 0, "lg2": 1, "rcp": 2, "ffma": 3, "ffma2": 4, "shfl": 5}
# shared-memory access patterns: SM clocks per warp-wide access (wavefronts)
SMEM_TESTS = {"ld128_uniform": 16, "ld128_quad_lane_mod4": 17, "ld128_lane_mod8": 18,
              "ld128_adjacent_pairs": 19, "ld128_adjacent_quads": 20, "ld128_adjacent_octets": 21,
              "ld128_distinct": 22, "ld64_uniform": 23, "ld64_distinct": 24, "ld32_uniform": 25,
              "ld32_distinct": 26, "st128_distinct": 27, "ld128_two_halves": 28}


def measure_pipes(warps=16, iters=4096, tests=PIPE_TESTS):
    """Per-SM rates from the pipe microbenchmark (one CTA per SM, fixed trip
    counts, the SM cycle counter around the loop): lane results per SM clock
    for the ALU tests, SM clocks per warp-wide access for the shared-memory
    ones.  Returns {name: rate} or None when the probe library is unavailable."""
    so = os.path.join(ROOT, "selective_state_space_114_b300", "libssprobe.so")
    if not os.path.exists(so):
        return None
    lib = ctypes.CDLL(so)
    lib.ssp_run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    out = {}
    for name, t in tests.items():
        c, r = ctypes.c_double(), ctypes.c_double()
        for _ in range(2):  # the first run loads the module
            if lib.ssp_run(t, warps, iters if t < 16 else iters // 4, ctypes.byref(c),
                           ctypes.byref(r)) != 0:
                return None
        out[name] = round(r.value, 3)
    return out


class Peaks:
    """Roofline denominators: FP32 and MUFU from per-SM rates x SMs x the
    maximum SM clock, HBM from the measured copy bandwidth."""

    def __init__(self, pipes=None):
        self.hbm_gbs, self.hbm_src = load_peaks()
        self.pipes_src = "measured" if pipes else "fallback"
        pipes = pipes or FALLBACK_PIPES
        self.fp32_per_clk = pipes["ffma"]
        self.mufu_per_clk = pipes["ex2"]
        self.fp32_t = SMS * self.fp32_per_clk * SM_MAX_MHZ * 1e6 / 1e12
        self.mufu_t = SMS * self.mufu_per_clk * SM_MAX_MHZ * 1e6 / 1e12
        self.pipes = pipes

    def describe(self):
        return {"hbm_gbs": self.hbm_gbs, "hbm": self.hbm_src,
                "fp32_tops": round(self.fp32_t, 2), "mufu_tops": round(self.mufu_t, 3),
                "pipes": self.pipes_src, "per_sm_clk": self.pipes,
                "clock_mhz": SM_MAX_MHZ, "sms": SMS}


# ---------------------------------------------------------------------------
# algorithmic work of the method (per scanned element)
# ---------------------------------------------------------------------------
def method_work(kind, s, Dch, N=N_STATE, Bsz=1):
    """Per scanned element (b, d, t) for kind in fwd, bwd, fwd_bwd; per token
    row (b, d) for step.  fp32 = FP32 add/mul/fma operations, mufu = exp / log
    / reciprocal evaluations, bytes = each tensor read or written once (B, C,
    dB, dC once per (b, t), parameters once).
      fwd:  per state delta*A, delta*u*B, the state update, C*h (4N); softplus
            4, D skip 1, delta*u 1, gate 3, the state sum 1; MUFU: N decays,
            softplus 2, sigmoid 2.  Bytes: u, delta, z in, y out, B and C.
      bwd:  (14N + 20) for forward and backward together, less the forward's
            4N + 10; MUFU N + 6.  Bytes: u, delta, z, dy in; du, ddelta, dz
            out; B, C in; dB, dC out (float32).
      step: a forward element with the state read and written (float32).
    """
    fwd = dict(fp32=4 * N + 10, mufu=N + 4, bytes=4 * s + 2 * N * s / Dch)
    bwd = dict(fp32=10 * N + 10, mufu=N + 6, bytes=7 * s + (2 * N * s + 8 * N) / Dch)
    if kind == "fwd":
        return fwd
    if kind == "bwd":
        return bwd
    if kind == "fwd_bwd":
        return {k: fwd[k] + bwd[k] for k in fwd}
    if kind == "step":
        return dict(fp32=4 * N + 10, mufu=N + 4, bytes=8 * N + 4 * s + 2 * N * s / Dch)
    raise ValueError(kind)


def roofline(work, units, ms, peaks, traffic=None):
    """The binding resource is the one whose algorithmic work takes longest at
    its peak; achieved = that work / the measured time."""
    t = ms * 1e-3
    times = {"hbm": work["bytes"] * units / (peaks.hbm_gbs * 1e9),
             "fp32": work["fp32"] * units / (peaks.fp32_t * 1e12),
             "mufu": work["mufu"] * units / (peaks.mufu_t * 1e12)}
    res = max(times, key=times.get)
    if res == "hbm":
        ach = work["bytes"] * units / t / 1e9
        out = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks.hbm_gbs, "unit": "GB/s"}
        frac = ach / peaks.hbm_gbs
    else:
        peak = peaks.fp32_t if res == "fp32" else peaks.mufu_t
        ach = work[res] * units / t / 1e12
        out = {"bound": "alu", "resource": res, "achieved": round(ach, 3),
               "peak": round(peak, 3), "unit": "TFLOP/s"}
        frac = ach / peak
    out["frac"] = round(frac, 4)
    out["traffic"] = traffic
    out["bound_ms"] = round(times[res] * 1e3, 4)
    return out


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
    return cfg, {
        "workload": "mamba130m-shaped layer 8x1536x2048 N=16: fwd + bwd + 1 decode token",
        "Bsz": cfg["Bsz"], "Dch": cfg["Dch"], "L": cfg["L"], "N": cfg["N"], "io_dtype": "bf16",
        "global_batch": cfg["Bsz"] * world,
        "parallelism": "replicas" if world == 1 else f"dp{world} (param-grad all-reduce)",
        "l2": "no flush: ~770 MiB of activations and gradients per step, 6x L2",
    }


# ---------------------------------------------------------------------------
# CPU (oracle) timing
# ---------------------------------------------------------------------------
def _host(cfg, n, seed, with_dy=False):
    """Host inputs of a workload cut to n channels (same distributions),
    widened exactly to float64."""
    x = synth.make_inputs(dict(cfg, Dch=n), seed=seed, with_dy=with_dy)
    return {k: synth.widen(v) for k, v in x.items()}


def oracle_pass(kind, cfg, n, seed):
    """One fp64 oracle pass over all batches x n channels x the full length
    (kind fwd, fwd_bwd or step: fwd + bwd + one decode token; decode: the
    configured number of successive steps over Bsz x n rows).  Returns
    (seconds, scanned elements)."""
    import oracle
    if kind == "decode":
        sub = dict(cfg, Dch=n, L=1)
        x = _host(sub, n, seed)
        toks = [{k: synth.widen(v) for k, v in synth.step_inputs(sub, k, seed=seed).items()}
                for k in range(cfg["steps"])]
        h = np.zeros((cfg["Bsz"], n, cfg["N"]))
        t0 = time.perf_counter()
        for tk in toks:
            _, h = oracle.step(h, tk["u"], tk["delta"], x["A"], tk["B"], tk["C"], x["D"], tk["z"],
                               x["delta_bias"], True)
        return time.perf_counter() - t0, cfg["Bsz"] * n * cfg["steps"]
    w = _host(cfg, n, seed, with_dy=kind != "fwd")
    t0 = time.perf_counter()
    _, h = oracle.scan_fwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                           w["delta_bias"], True)
    if kind != "fwd":
        oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w["D"], w["z"],
                        w["delta_bias"], True, w["dy"])
    if kind == "step":
        sub = dict(cfg, Dch=n, L=1)
        tk = {k: synth.widen(v) for k, v in synth.step_inputs(sub, 0, seed=seed).items()}
        oracle.step(h, tk["u"], tk["delta"], w["A"], tk["B"], tk["C"], w["D"], tk["z"],
                    w["delta_bias"], True)
    return time.perf_counter() - t0, cfg["Bsz"] * n * cfg["L"]


def oracle_sample(kind, cfg, seed, target_s):
    """The oracle as it stands on the host cores, on about target_s seconds of
    the workload (whole channels, all batches, full length), sized by doubling
    the channel count."""
    import oracle
    n = min(cfg["Dch"], 2)
    while True:
        t, e = oracle_pass(kind, cfg, n, seed)
        if t >= 0.5 * target_s or n >= cfg["Dch"]:
            break
        n = int(min(cfg["Dch"], max(n + 1, n * min(8.0, target_s / max(t, 1e-3)))))
    steps = f"{cfg['steps']} steps of " if kind == "decode" else ""
    return {"value": round(e / t / 1e9, 6), "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle", "sample": f"fp64 {kind}: {steps}{cfg['Bsz']} x {n} of {cfg['Dch']} "
                                        f"channels x L={cfg['L']} ({e} el, {t:.1f} s)",
            "short": f"{steps}{cfg['Bsz']}x{n}x{cfg['L']}, {t:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    cfg, conf = workload_config(1)
    if rank != 0:
        return 0
    import oracle
    cores = oracle.default_threads()
    W, K = max(3, args.warmup), args.steps
    per_step = max(0.5, 150.0 / (W + K))  # the whole run in about 150 s
    n = 2
    while True:
        t, e = oracle_pass("step", cfg, n, cfg["seed"])
        if t >= 0.5 * per_step or n >= cfg["Dch"]:
            break
        n = int(min(cfg["Dch"], max(n + 1, n * per_step / max(t, 1e-3))))
    for _ in range(W):
        oracle_pass("step", cfg, n, cfg["seed"])
    times = [oracle_pass("step", cfg, n, cfg["seed"])[0] for _ in range(K)]
    elems = cfg["Bsz"] * n * cfg["L"]
    ms = 1e3 * sum(times) / K
    value = elems / (ms * 1e-3) / 1e9
    sample = (f"each step: fp64 oracle fwd + bwd + 1 decode token over {cfg['Bsz']} x {n} of "
              f"{cfg['Dch']} channels x L={cfg['L']} ({elems} elements)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": conf,
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU timing
# ---------------------------------------------------------------------------
def _timed_ms(fns, steps, dev, flush=False):
    """Mean device time of each function over `steps` rounds after 3 warm-up
    rounds.  The GPU first spins (~25 ms) so that the host has enqueued every
    timed launch before the first runs.  flush: a 256 MiB read before each
    round empties L2 of the round's data (for workloads smaller than L2)."""
    import torch
    buf = torch.ones(64 * 2 ** 20, device=dev, dtype=torch.float32) if flush else None
    sink = torch.empty((), device=dev, dtype=torch.float32)
    for _ in range(3):
        for f in fns:
            f()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)
    for row in evs:
        if buf is not None:
            torch.sum(buf, dim=0, out=sink)
        row[0].record()
        for i, f in enumerate(fns):
            f()
            row[i + 1].record()
    torch.cuda.synchronize()
    return [statistics.mean(r[i].elapsed_time(r[i + 1]) for r in evs) for i in range(len(fns))]


def _device_inputs(cfg, dev, seed, with_dy=False):
    """Inputs drawn on the device by torch's seeded generator with the
    workload's distributions (timing does not depend on the values); A, D
    and delta_bias from the host generator."""
    import torch
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    dtype = {"bf16": torch.bfloat16, "f16": torch.float16}.get(cfg["dtype"], torch.float32)
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


def _grads(x, dev):
    import torch
    Bsz, Dch, L = x["u"].shape
    N = x["A"].shape[1]
    return {"du": torch.empty_like(x["u"]), "ddelta": torch.empty_like(x["u"]),
            "dz": torch.empty_like(x["u"]), "dA": torch.empty((Dch, N), device=dev),
            "dB": torch.empty((Bsz, N, L), device=dev), "dC": torch.empty((Bsz, N, L), device=dev),
            "dD": torch.empty((Dch,), device=dev), "ddelta_bias": torch.empty((Dch,), device=dev)}


BWD_STAGES = ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce")


def _r(d):
    """The roofline keys a config entry keeps: the binding resource and the
    fraction of its peak (the peaks are in the line's "peaks")."""
    return {"bound": d.get("resource", d["bound"]), "frac": d["frac"]}


def config_lines(ss, dev, seed, peaks, cpu=True):
    """One entry per workload of the configuration list: time, Gelem/s,
    roofline (method counts), and the oracle on a bounded sample."""
    import torch
    out = {}
    # Mamba-130M-shaped layer, forward (bf16)
    cfg = synth.config(1)
    x, _ = _device_inputs(cfg, dev, seed + 1)
    E = cfg["Bsz"] * cfg["Dch"] * cfg["L"]
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y = torch.empty_like(x["u"])
    (t,) = _timed_ms([lambda: ss.ss_scan_fwd(*args, out=y)], 20, dev)
    out["mamba130m_fwd"] = {"ms": round(t, 4),
                            "gelem_s": round(E / t / 1e6, 2),
                            **_r(roofline(method_work("fwd", 2, cfg["Dch"]), E, t, peaks))}
    del x, y
    # Mamba-370M-shaped layer, forward + backward (fp32)
    cfg = synth.config(2)
    x, _ = _device_inputs(cfg, dev, seed + 2, with_dy=True)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y, g = torch.empty_like(x["u"]), _grads(x, dev)
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_F32), device=dev,
                     dtype=torch.uint8)
    fns = [lambda: ss.ss_scan_fwd(*args, out=y, save_to=ws)] + [
        lambda st=st: ss.ss_scan_bwd(*args, x["dy"], workspace=ws, out=g, stages=(st,),
                                     saved=True)
        for st in BWD_STAGES]
    ms = _timed_ms(fns, 10, dev)
    tb = sum(ms[1:])
    out["mamba370m_fwd_bwd"] = {
        "ms": round(sum(ms), 4),
        "gelem_s": round(E / sum(ms) / 1e6, 2),
        **_r(roofline(method_work("fwd_bwd", 4, Dch), E, sum(ms), peaks)),
        "fwd": {"ms": round(ms[0], 4), "frac": roofline(method_work("fwd", 4, Dch), E, ms[0],
                                                        peaks)["frac"]},
        "bwd": {"ms": round(tb, 4), "frac": roofline(method_work("bwd", 4, Dch), E, tb,
                                                     peaks)["frac"],
                "stages": [round(v, 4) for v in ms[1:]]}}
    del x, y, g, ws
    torch.cuda.empty_cache()
    # long sequence, forward (bf16)
    cfg = synth.config(3)
    x, _ = _device_inputs(cfg, dev, seed + 3)
    E = cfg["Bsz"] * cfg["Dch"] * cfg["L"]
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y = torch.empty_like(x["u"])
    h = torch.empty((cfg["Bsz"], cfg["Dch"], cfg["N"]), device=dev)
    (t,) = _timed_ms([lambda: ss.ss_scan_fwd(*args, out=y, h_last=h, return_last_state=True)],
                     5, dev)
    out["long_sequence_fwd"] = {"ms": round(t, 4),
                                "gelem_s": round(E / t / 1e6, 2),
                                **_r(roofline(method_work("fwd", 2, cfg["Dch"]), E, t, peaks))}
    del x, y, h
    torch.cuda.empty_cache()
    # decode: 128 successive tokens, the state updated in place (L2 flushed
    # before each run of 128; within a run the 84 MB state may stay in L2)
    cfg = synth.config(4)
    Bsz, Dch, N, S = cfg["Bsz"], cfg["Dch"], cfg["N"], cfg["steps"]
    x, _ = _device_inputs(dict(cfg, L=1), dev, seed + 4)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 40)
    bf = torch.bfloat16
    toks = [{k: torch.randn(shp, generator=gen, device=dev).to(bf) for k, shp in
             (("u", (Bsz, Dch)), ("delta", (Bsz, Dch)), ("z", (Bsz, Dch)), ("B", (Bsz, N)),
              ("C", (Bsz, N)))} for _ in range(S)]
    h = torch.zeros((Bsz, Dch, N), device=dev)
    ys = torch.empty((S, Bsz, Dch), device=dev, dtype=bf)

    def run128():
        for i, tk in enumerate(toks):
            ss.ss_step(h, tk["u"], tk["delta"], x["A"], tk["B"], tk["C"], x["D"], tk["z"],
                       x["delta_bias"], True, out=ys[i])

    (t,) = _timed_ms([run128], 5, dev, flush=True)
    units = Bsz * Dch * S
    out["decode_128_steps"] = {"ms": round(t, 4), "us_per_token": round(1e3 * t / S, 2),
                               "gelem_s": round(units / t / 1e6, 2),
                               **_r(roofline(method_work("step", 2, Dch), units, t, peaks))}
    del x, toks, h, ys
    torch.cuda.empty_cache()
    if cpu:
        kinds = {"mamba130m_fwd": ("fwd", 1), "mamba370m_fwd_bwd": ("fwd_bwd", 2),
                 "long_sequence_fwd": ("fwd", 3), "decode_128_steps": ("decode", 4)}
        for key, (kind, ci) in kinds.items():
            c = synth.config(ci)
            o = oracle_sample(kind, c, c["seed"], target_s=3.0)
            out[key]["cpu"] = {"gelem_s": o["value"], "cores": o["cores"], "sample": o["short"]}
    return out


def next_rows(ss, dev, seed, peaks):
    """The block's producers of the scan inputs on the bench layer's shape
    (8 x 1536 x 2048, bf16), L2 flushed before each call: causal conv1d
    (width 4) + silu forward and backward, and the input projection (x_proj
    then dt_proj, dt_rank 48, on the tensor cores).  HBM-bound."""
    import torch
    cfg = synth.config(CFG_INDEX)
    Bsz, Dch, L, N, K, R = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"], 4, 48
    E = Bsz * Dch * L
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 7)
    bf = torch.bfloat16
    rnd = lambda *s: torch.randn(s, generator=gen, device=dev)
    x, g = rnd(Bsz, Dch, L).to(bf), rnd(Bsz, Dch, L).to(bf)
    w, b = rnd(Dch, K) / 2.0, rnd(Dch)
    u = torch.empty_like(x)
    grads = {"dx": torch.empty_like(x), "dw": torch.empty((Dch, K), device=dev),
             "dbias": torch.empty((Dch,), device=dev)}
    Wx = (rnd(R + 2 * N, Dch) / Dch ** 0.5).to(bf)
    Wdt = (rnd(Dch, R) / R ** 0.5).to(bf)
    xo = (torch.empty_like(x), torch.empty((Bsz, N, L), device=dev, dtype=bf),
          torch.empty((Bsz, N, L), device=dev, dtype=bf))
    ms = [_timed_ms([f], 16, dev, flush=True)[0] for f in (
        lambda: ss.ss_conv1d_silu(x, w, b, True, out=u),
        lambda: ss.ss_conv1d_silu_bwd(x, w, b, True, g, out=grads),
        lambda: ss.ss_xproj(x, Wx, Wdt, N, out=xo))]
    nbytes = (2 * 2 * E, 3 * 2 * E,
              2 * E * 2 + 2 * 2 * Bsz * N * L + 2 * (R + 2 * N) * Dch + 2 * Dch * R)
    res = {}
    for name, t, nb in zip(("conv1d_silu_fwd", "conv1d_silu_bwd", "xproj"), ms, nbytes):
        ach = nb / (t * 1e-3) / 1e9
        res[name] = {"ms": round(t, 4), "bound": "hbm", "frac": round(ach / peaks.hbm_gbs, 4)}
    flops = 2 * Bsz * L * Dch * (R + 2 * N) + 2 * Bsz * L * R * Dch
    res["xproj"]["tensor_tflops"] = round(flops / (ms[2] * 1e-3) / 1e12, 2)
    res["xproj"]["device_errors"] = ss.ss_check_device_errors()
    del x, g, u, grads, xo
    res.update(scan_variants(ss, dev, seed, peaks))
    return res


def scan_variants(ss, dev, seed, peaks):
    """The scan's other configurations on the bench layer's shape (8 x 1536 x
    2048), inputs larger than L2 timed back to back: state size 64 (forward,
    and the backward with the chunk states kept by the forward), fp16 I/O
    (forward), and a chunked prefill (the forward in 4 pieces of 512 steps,
    each continuing from the state the previous piece left)."""
    import torch
    res = {}
    base = synth.config(CFG_INDEX)
    # state size 64
    cfg = dict(base, N=64)
    x, _ = _device_inputs(cfg, dev, seed + 11, with_dy=True)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    E = Bsz * Dch * L
    a = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y, g = torch.empty_like(x["u"]), _grads(x, dev)
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_BF16), device=dev,
                     dtype=torch.uint8)
    tf, tb = _timed_ms([lambda: ss.ss_scan_fwd(*a, out=y, save_to=ws),
                        lambda: ss.ss_scan_bwd(*a, x["dy"], workspace=ws, out=g, saved=True)],
                       10, dev)
    res["state_size_64_fwd"] = {"ms": round(tf, 4), "gelem_s": round(E / tf / 1e6, 2),
                                **_r(roofline(method_work("fwd", 2, Dch, N), E, tf, peaks))}
    res["state_size_64_bwd"] = {"ms": round(tb, 4), "gelem_s": round(E / tb / 1e6, 2),
                                **_r(roofline(method_work("bwd", 2, Dch, N), E, tb, peaks))}
    del x, y, g, ws
    # fp16 I/O and chunked prefill (16 states)
    cfg = dict(base, dtype="f16")
    x, _ = _device_inputs(cfg, dev, seed + 12)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    a = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y = torch.empty_like(x["u"])
    (t16,) = _timed_ms([lambda: ss.ss_scan_fwd(*a, out=y)], 10, dev)
    res["fp16_fwd"] = {"ms": round(t16, 4), "gelem_s": round(E / t16 / 1e6, 2),
                       **_r(roofline(method_work("fwd", 2, Dch, N), E, t16, peaks))}
    xb, _ = _device_inputs(base, dev, seed + 13)
    pieces, P = 4, L // 4
    parts = [{k: xb[k][..., i * P:(i + 1) * P].contiguous() for k in ("u", "delta", "z", "B", "C")}
             for i in range(pieces)]
    yp = [torch.empty_like(pp["u"]) for pp in parts]
    h = torch.empty((Bsz, Dch, N), device=dev)

    def prefill():
        for i, pp in enumerate(parts):
            ss.ss_scan_fwd(pp["u"], pp["delta"], xb["A"], pp["B"], pp["C"], xb["D"], pp["z"],
                           xb["delta_bias"], True, out=yp[i], h_last=h, return_last_state=True,
                           h0=h if i else None)
    (tp,) = _timed_ms([prefill], 10, dev)
    res["chunked_prefill_4x512"] = {"ms": round(tp, 4), "gelem_s": round(E / tp / 1e6, 2),
                                    **_r(roofline(method_work("fwd", 2, Dch, N), E, tp, peaks))}
    return res


# The sources each timed kernel is built from: its ncu figures are reported
# only while their code (comments and blank lines aside) is unchanged.
KERNEL_SOURCES = {"fwd": ("common.cuh", "launch.h", "scan_fwd.cu"),
                  "bwd_states": ("common.cuh", "launch.h", "scan_bwd.cu"),
                  "bwd_reverse": ("common.cuh", "launch.h", "scan_bwd.cu")}


def _code_only(text):
    """C++ source without its comments and blank lines, runs of spaces in a
    line collapsed to one."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(l.split()) for l in text.splitlines() if l.strip())


def csrc_digest(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(ROOT, "selective_state_space_114_b300", "csrc", name)).read()
        h.update(_code_only(src).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, when it was
    taken on the current kernel sources; else None."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    except Exception:
        return None
    v = d.get("kernels", {}).get(kernel)
    if v is None or kernel not in KERNEL_SOURCES or v.get("csrc_digest") != csrc_digest(kernel):
        return None
    return v.get("dram_bytes_per_launch")


def run_profile_workload(args):
    """Run one workload's kernels --profile-iters times and exit (for an ncu
    capture): mamba130m (bf16 8 x 1536 x L, fwd + bwd), mamba370m (fp32 8 x
    2048 x L, fwd + bwd), long_sequence (bf16 1 x 5120 x L forward), decode
    (one token on 256 x 5120), producers (conv1d + silu fwd and bwd and the
    input projection on bf16 8 x 1536 x L); --profile-L cuts L to keep a
    capture small."""
    import torch
    import selective_state_space_114_b300 as ss
    dev = torch.device("cuda", 0)
    if args.profile_workload in ("decode", "producers"):
        return _profile_other(args, ss, dev)
    ci = {"mamba130m": 1, "mamba370m": 2, "long_sequence": 3}[args.profile_workload]
    cfg = synth.config(ci)
    if args.profile_L:
        cfg = dict(cfg, L=args.profile_L)
    bwd = ci in (1, 2)
    x, _ = _device_inputs(cfg, dev, cfg["seed"], with_dy=bwd)
    Bsz, Dch, L, N = cfg["Bsz"], cfg["Dch"], cfg["L"], cfg["N"]
    a = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True)
    y, h = torch.empty_like(x["u"]), torch.empty((Bsz, Dch, N), device=dev)
    ws = None
    if bwd:
        code = ss.SS_BF16 if cfg["dtype"] == "bf16" else ss.SS_F32
        ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, code), device=dev,
                         dtype=torch.uint8)
    for _ in range(args.profile_iters):
        ss.ss_scan_fwd(*a, out=y, h_last=h, return_last_state=True, save_to=ws)
        if ws is not None:
            ss.ss_scan_bwd(*a, x["dy"], workspace=ws, saved=True)
    torch.cuda.synchronize()
    print(json.dumps({"profile_workload": args.profile_workload, "Bsz": Bsz, "Dch": Dch, "L": L,
                      "iters": args.profile_iters}))
    return 0


def _profile_other(args, ss, dev):
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    bf = torch.bfloat16
    rnd = lambda *s: torch.randn(s, generator=gen, device=dev)
    if args.profile_workload == "decode":
        cfg = synth.config(4)
        Bsz, Dch, N = cfg["Bsz"], cfg["Dch"], cfg["N"]
        x, _ = _device_inputs(dict(cfg, L=1), dev, cfg["seed"])
        tk = {k: rnd(*shp).to(bf) for k, shp in (("u", (Bsz, Dch)), ("delta", (Bsz, Dch)),
                                                ("z", (Bsz, Dch)), ("B", (Bsz, N)),
                                                ("C", (Bsz, N)))}
        h = torch.zeros((Bsz, Dch, N), device=dev)
        for _ in range(args.profile_iters):
            ss.ss_step(h, tk["u"], tk["delta"], x["A"], tk["B"], tk["C"], x["D"], tk["z"],
                       x["delta_bias"], True)
        shape = {"Bsz": Bsz, "Dch": Dch}
    else:
        cfg = synth.config(CFG_INDEX)
        Bsz, Dch, L, N, K, R = (cfg["Bsz"], cfg["Dch"], args.profile_L or cfg["L"], cfg["N"],
                                4, 48)
        x, g = rnd(Bsz, Dch, L).to(bf), rnd(Bsz, Dch, L).to(bf)
        w, b = rnd(Dch, K) / 2.0, rnd(Dch)
        Wx, Wdt = (rnd(R + 2 * N, Dch) / Dch ** 0.5).to(bf), (rnd(Dch, R) / R ** 0.5).to(bf)
        for _ in range(args.profile_iters):
            ss.ss_conv1d_silu(x, w, b, True)
            ss.ss_conv1d_silu_bwd(x, w, b, True, g)
            ss.ss_xproj(x, Wx, Wdt, N)
        shape = {"Bsz": Bsz, "Dch": Dch, "L": L}
    torch.cuda.synchronize()
    print(json.dumps({"profile_workload": args.profile_workload, **shape,
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
    peaks = Peaks(measure_pipes() if rank == 0 else None)
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
    g = _grads(d, dev)
    ws = torch.empty(ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, ss.SS_BF16), device=dev,
                     dtype=torch.uint8)
    yt = torch.empty((Bsz, Dch), device=dev, dtype=bf)
    names = ["fwd", "bwd_states", "bwd_reverse", "bwd_reduce", "step"]

    def one_step(evs=None, bufs=None):
        """One pass of the path on the current stream; bufs = (inputs, token,
        outputs, state) of an end-to-end buffer set, else the resident ones."""
        dd, tk, out, hh = bufs if bufs is not None else (d, dt, dict(y=y, yt=yt, **g), h)
        gg = {k: out[k] for k in g}
        rec = (lambda i: evs[i].record()) if evs is not None else (lambda i: None)
        rec(0)
        ss.ss_scan_fwd(dd["u"], dd["delta"], dd["A"], dd["B"], dd["C"], dd["D"], dd["z"],
                       dd["delta_bias"], True, return_last_state=True, out=out["y"], h_last=hh,
                       save_to=ws)
        rec(1)
        for i, st in enumerate(BWD_STAGES):
            ss.ss_scan_bwd(dd["u"], dd["delta"], dd["A"], dd["B"], dd["C"], dd["D"], dd["z"],
                           dd["delta_bias"], True, dd["dy"], workspace=ws, out=gg, stages=(st,),
                           saved=True)
            rec(2 + i)
        ss.ss_step(hh, tk["u"], tk["delta"], dd["A"], tk["B"], tk["C"], dd["D"], tk["z"],
                   dd["delta_bias"], True, out=out["yt"])
        rec(5)
        if world > 1:
            sdist.allreduce_param_grads(gg)

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
        # the GPU spins first (about 12 ms + 1.2 ms per step) so that the host
        # has enqueued the timed steps before the first one runs: the events
        # then see device time only, not the host's launch rate
        torch.cuda._sleep(25_000_000 + 2_500_000 * K)
        start.record()
        for k in range(K):
            one_step(evs[k])
        end.record()
        torch.cuda.synchronize()
    barrier()
    ms_local = start.elapsed_time(end) / K
    ms = sdist.max_over_ranks(ms_local, device=dev)
    per = {nm: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(K))
           for i, nm in enumerate(names)}
    value = world * E / (ms * 1e-3) / 1e9

    side = rank == 0 and not args.step_only
    # the first backward stage when the chunk states are recomputed (the
    # backward without a saving forward): summaries and carries of both
    (t_states_recomputed,) = _timed_ms(
        [lambda: ss.ss_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                d["delta_bias"], True, d["dy"], workspace=ws, out=g,
                                stages=("ss_scan_bwd_states",))], 10, dev) if side else (None,)
    configs = config_lines(ss, dev, seed, peaks, cpu=not args.no_cpu_baseline) if side else None
    nxt = next_rows(ss, dev, seed, peaks) if side else None

    # end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and its outputs back out.  The
    # steps are pipelined over three streams (copy in, compute, copy out) with
    # two buffer sets, so the copies of one step overlap the kernels of
    # another and the two copy directions overlap each other.
    Ke = max(4, min(K, 10))
    outs = {"y": y, "yt": yt, **g}
    sets = [({k: torch.empty_like(v) for k, v in d.items()},
             {k: torch.empty_like(v) for k, v in dt.items()},
             {k: torch.empty_like(v) for k, v in outs.items()},
             torch.empty_like(h)) for _ in range(2)]
    hout = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
            for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in list(hx.values()) + list(ht.values()))
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    s_comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = ([ev() for _ in range(Ke)] for _ in range(3))
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(Ke):
        dd, tk, out, hh = sets[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(comp_done[k - 2])  # the set's inputs are free again
            for n, v in hx.items():
                dd[n].copy_(v, non_blocking=True)
            for n, v in ht.items():
                tk[n].copy_(v, non_blocking=True)
            in_done[k].record(s_in)
        s_comp.wait_event(in_done[k])
        if k >= 2:
            s_comp.wait_event(out_done[k - 2])  # the set's outputs have been read out
        one_step(bufs=(dd, tk, out, hh))
        comp_done[k].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            for n, v in out.items():
                hout[k % 2][n].copy_(v, non_blocking=True)
            out_done[k].record(s_out)
    s_comp.wait_event(out_done[Ke - 1])
    e1.record(s_comp)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = sdist.max_over_ranks(e0.elapsed_time(e1) / Ke, device=dev)
    del sets

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    work = {"fwd": method_work("fwd", 2, Dch), "bwd_reverse": method_work("bwd", 2, Dch)}
    kernels = {}
    for nm in names:
        kernels[nm] = {"ms": round(per[nm], 4), "share": round(per[nm] / sum(per.values()), 4)}
        if nm in work:
            r = roofline(work[nm], E, per[nm], peaks)
            kernels[nm].update(frac=r["frac"], bound=r.get("resource", r["bound"]))
    rstep = roofline(method_work("step", 2, Dch), Bsz * Dch, per["step"], peaks)
    kernels["step"].update(frac=rstep["frac"], bound="hbm")
    tb = per["bwd_states"] + per["bwd_reverse"] + per["bwd_reduce"]
    rbwd = roofline(method_work("bwd", 2, Dch), E, tb, peaks)
    dominant = max(("fwd", "bwd_reverse"), key=lambda nm: per[nm])
    top = roofline(work[dominant], E, per[dominant], peaks, ncu_traffic(dominant))
    top.pop("bound_ms", None)
    # the standard keys first; the per-kernel and per-workload detail last
    # (a reader of the line's tail sees it)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": conf,
        "gpu_launches": K * LAUNCHES_PER_STEP,
        "e2e": {"value": round(world * E / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 3)},
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample("step", cfg, seed, target_s=12.0)
        cb.pop("short")
        line["cpu_baseline"] = cb
    pk = peaks.describe()
    pk.pop("per_sm_clk")
    line.update({
        "peaks": pk,
        "next_rows": nxt,
        "roofline": {"kernel": dominant, **top},
        "configs": configs,
        "backward": {"ms": round(tb, 4), "frac": rbwd["frac"], "bound": rbwd.get("resource"),
                     "states_stage_when_recomputed_ms": (round(t_states_recomputed, 4)
                                                         if t_states_recomputed else None)},
        "kernels": kernels,
    })
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
                    help="skip the oracle timings on the host cores")
    ap.add_argument("--step-only", action="store_true",
                    help="time the headline step only (no per-workload or producer entries)")
    ap.add_argument("--pipes", action="store_true",
                    help="print the pipe microbenchmark's per-SM rates and exit")
    ap.add_argument("--profile-workload",
                    choices=["mamba130m", "mamba370m", "long_sequence", "decode", "producers"],
                    help="only run that workload's kernels (for an ncu capture) and exit")
    ap.add_argument("--profile-L", type=int, default=0)
    ap.add_argument("--profile-iters", type=int, default=2)
    args = ap.parse_args()
    if args.pipes:
        import torch
        torch.cuda.set_device(0)
        rates = measure_pipes()
        smem = measure_pipes(tests=SMEM_TESTS)
        print(json.dumps({"per_sm_per_clock": rates, "smem_clocks_per_access": smem,
                          "peaks": Peaks(rates).describe(), "gpu": torch.cuda.get_device_name(0)}))
        return 0 if rates else 1
    if args.profile_workload:
        return run_profile_workload(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
