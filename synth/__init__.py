"""Seeded synthetic inputs for the selective scan, shared by the tests,
the bench and the oracle checks.

This module holds no arithmetic of the scan itself.  It turns
(seed, tensor id, element index) into pseudo-random numbers with a
counter-based generator (splitmix64 + Box-Muller, implemented in
``synth.c``), so that one (batch, channel) row of even the largest
workload can be regenerated on its own, and it rounds to bf16 with
round-to-nearest-even so that both sides consume identical values.

bf16 tensors are returned as ``numpy.uint16`` bit patterns; ``widen``
turns them (or float32 arrays) into exact float64 copies.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import CONFIGS, TENSOR_IDS, config  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (gcc, -O2)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            l = ctypes.CDLL(_SO)
            u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
            l.synth_normal_f32.argtypes = [u64, u64, p, i64, i64, p]
            l.synth_normal_bf16.argtypes = [u64, u64, p, i64, i64, p]
            l.synth_uniform_f64.argtypes = [u64, u64, i64, i64, p]
            l.synth_f32_to_bf16.argtypes = [p, i64, p]
            for f in (l.synth_normal_f32, l.synth_normal_bf16, l.synth_uniform_f64, l.synth_f32_to_bf16):
                f.restype = None
            _lib = l
    return _lib


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))
    return _POOL


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, tid: int, count: int, dtype: str = "f32", start: int = 0) -> np.ndarray:
    """N(0,1) samples for element indices start .. start+count-1 of tensor ``tid``.

    dtype "f32" -> float32 array; "bf16" -> uint16 bf16 bit patterns;
    "f16" -> float16 array (the float32 samples rounded to nearest even).
    """
    l = lib()
    if dtype == "f16":
        return normal(seed, tid, count, "f32", start).astype(np.float16)
    if dtype == "f32":
        out = np.empty(count, np.float32)
        fn = l.synth_normal_f32
        es = 4
    elif dtype == "bf16":
        out = np.empty(count, np.uint16)
        fn = l.synth_normal_bf16
        es = 2
    else:
        raise ValueError(dtype)
    step = 1 << 22
    if count <= step:
        fn(seed, tid, None, start, count, _ptr(out))
        return out
    base = _ptr(out)
    futs = [
        _pool().submit(fn, seed, tid, None, start + k, min(step, count - k), base + k * es)
        for k in range(0, count, step)
    ]
    for f in futs:
        f.result()
    return out


def normal_at(seed: int, tid: int, idx: np.ndarray, dtype: str = "f32") -> np.ndarray:
    """N(0,1) samples at arbitrary flat element indices ``idx``."""
    l = lib()
    idx = np.ascontiguousarray(idx, dtype=np.int64).ravel()
    if dtype == "f16":
        return normal_at(seed, tid, idx, "f32").astype(np.float16)
    if dtype == "f32":
        out = np.empty(idx.size, np.float32)
        l.synth_normal_f32(seed, tid, _ptr(idx), 0, idx.size, _ptr(out))
    elif dtype == "bf16":
        out = np.empty(idx.size, np.uint16)
        l.synth_normal_bf16(seed, tid, _ptr(idx), 0, idx.size, _ptr(out))
    else:
        raise ValueError(dtype)
    return out


def uniform(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """Uniform (0, 1) float64 samples for indices start .. start+count-1."""
    out = np.empty(count, np.float64)
    lib().synth_uniform_f64(seed, tid, start, count, _ptr(out))
    return out


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().synth_f32_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def to_f16(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (nearest even)."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16)


def widen(x: np.ndarray) -> np.ndarray:
    """Exact float64 copy of a float32 or float16 array or of bf16 bit patterns (uint16)."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Per-tensor recipes.  Parameters (A, D, delta_bias) depend on the channel d
# only; activations are [Bsz][Dch][L], B and C are [Bsz][N][L].
# ---------------------------------------------------------------------------

def param_A(Dch: int, N: int) -> np.ndarray:
    """A[d, n] = -(n + 1) (S4D-real initialisation), float32 [Dch][N]."""
    return np.ascontiguousarray(np.broadcast_to(-(np.arange(N, dtype=np.float32) + 1.0), (Dch, N)))


def param_D(seed: int, Dch: int) -> np.ndarray:
    return normal(seed, TENSOR_IDS["D"], Dch, "f32")


def param_delta_bias(seed: int, Dch: int, dt_range) -> np.ndarray:
    """delta_bias = inverse softplus of dt, dt log-uniform in dt_range (float32)."""
    lo, hi = dt_range
    uu = uniform(seed, TENSOR_IDS["dt"], Dch)
    dt = np.exp(np.log(lo) + uu * (np.log(hi) - np.log(lo)))
    return np.log(np.expm1(dt)).astype(np.float32)


def make_inputs(cfg: dict, seed: int | None = None, with_dy: bool = False, **shape) -> dict:
    """All scan inputs of a workload as host numpy arrays.

    ``shape`` may override Bsz/Dch/L/N (smaller parity cases with the same
    distributions).  Activations and B/C come back in the workload dtype
    (float32, or bf16 bit patterns); A, D, delta_bias are float32.
    """
    c = dict(cfg)
    c.update(shape)
    seed = c["seed"] if seed is None else seed
    Bsz, Dch, L, N, dt = c["Bsz"], c["Dch"], c["L"], c["N"], c["dtype"]
    E = Bsz * Dch * L
    out = {
        "u": normal(seed, TENSOR_IDS["u"], E, dt).reshape(Bsz, Dch, L),
        "delta": normal(seed, TENSOR_IDS["delta"], E, dt).reshape(Bsz, Dch, L),
        "z": normal(seed, TENSOR_IDS["z"], E, dt).reshape(Bsz, Dch, L),
        "B": normal(seed, TENSOR_IDS["B"], Bsz * N * L, dt).reshape(Bsz, N, L),
        "C": normal(seed, TENSOR_IDS["C"], Bsz * N * L, dt).reshape(Bsz, N, L),
        "A": param_A(Dch, N),
        "D": param_D(seed, Dch),
        "delta_bias": param_delta_bias(seed, Dch, c["dt_range"]),
    }
    if with_dy:
        out["dy"] = normal(seed, TENSOR_IDS["dy"], E, dt).reshape(Bsz, Dch, L)
    return out


def row_inputs(cfg: dict, b: int, d: int, seed: int | None = None) -> dict:
    """The inputs one (b, d) row of a workload needs, regenerated on their own:
    u/delta/z rows [L], B/C [N][L] of batch b, A[d] [N], D[d], delta_bias[d]."""
    seed = cfg["seed"] if seed is None else seed
    Dch, L, N, dt = cfg["Dch"], cfg["L"], cfg["N"], cfg["dtype"]
    r0 = (b * Dch + d) * L
    bc0 = b * N * L
    return {
        "u": normal(seed, TENSOR_IDS["u"], L, dt, start=r0),
        "delta": normal(seed, TENSOR_IDS["delta"], L, dt, start=r0),
        "z": normal(seed, TENSOR_IDS["z"], L, dt, start=r0),
        "B": normal(seed, TENSOR_IDS["B"], N * L, dt, start=bc0).reshape(N, L),
        "C": normal(seed, TENSOR_IDS["C"], N * L, dt, start=bc0).reshape(N, L),
        "A": param_A(Dch, N)[d],
        "D": param_D(seed, Dch)[d : d + 1],
        "delta_bias": param_delta_bias(seed, Dch, cfg["dt_range"])[d : d + 1],
    }


def step_inputs(cfg: dict, k: int, seed: int | None = None) -> dict:
    """Per-token inputs of decode step k: u/delta/z [Bsz][Dch], B/C [Bsz][N]."""
    seed = cfg["seed"] if seed is None else seed
    Bsz, Dch, N, dt = cfg["Bsz"], cfg["Dch"], cfg["N"], cfg["dtype"]
    base = 1000 + 16 * k
    return {
        "u": normal(seed, base + TENSOR_IDS["u"], Bsz * Dch, dt).reshape(Bsz, Dch),
        "delta": normal(seed, base + TENSOR_IDS["delta"], Bsz * Dch, dt).reshape(Bsz, Dch),
        "z": normal(seed, base + TENSOR_IDS["z"], Bsz * Dch, dt).reshape(Bsz, Dch),
        "B": normal(seed, base + TENSOR_IDS["B"], Bsz * N, dt).reshape(Bsz, N),
        "C": normal(seed, base + TENSOR_IDS["C"], Bsz * N, dt).reshape(Bsz, N),
    }
