"""fp64 CPU oracle of the selective scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it, and it shares no code
with that path.

All functions take float64 numpy arrays (callers widen bf16/float32 inputs
exactly beforehand) and return float64 arrays.  The arithmetic lives in
``oracle.c``; this file only marshals arguments.  See that file's header
for what is computed and which passages of the pages it follows.

Parity pins (tests/test_oracle_pins.py) tie every function here to
something other than itself: a brute-force closed form, a textbook IIR
filter (scipy.signal.lfilter), invariants, the Blelloch-ordered variant and
central finite differences.  ``Oracle(path)`` binds any build of
``oracle.c`` (the pin tests also run against deliberately mutated builds
to show that each pin can fail).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_c(src: str, out: str) -> str:
    """gcc -O2 (IEEE fp64, no fast-math, no FMA contraction on x86-64)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(SOURCE):
        compile_c(SOURCE, _SO)
    return _SO


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(x, shape=None):
    if x is None:
        return None
    a = np.ascontiguousarray(x, dtype=np.float64)
    if shape is not None and a.shape != tuple(shape):
        a = a.reshape(shape)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


class Oracle:
    """Binding of one build of oracle.c."""

    def __init__(self, path: str):
        l = ctypes.CDLL(path)
        p, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        l.oracle_scan_fwd.argtypes = [p] * 8 + [ci, i64, i64, i64, i64, p, p, p, ci]
        l.oracle_scan_fwd_blelloch.argtypes = l.oracle_scan_fwd.argtypes
        l.oracle_scan_bwd.argtypes = [p] * 8 + [ci, i64, i64, i64, i64] + [p] * 9 + [ci]
        l.oracle_step.argtypes = [p] * 9 + [ci, i64, i64, i64, p, ci]
        l.oracle_conv1d_silu.argtypes = [p] * 3 + [ci, i64, i64, i64, i64, p, ci]
        l.oracle_conv1d_silu_bwd.argtypes = [p] * 3 + [ci, p, i64, i64, i64, i64, p, p, p, ci]
        l.oracle_xproj.argtypes = [p] * 3 + [i64] * 5 + [p] * 3 + [ci]
        for f in (l.oracle_scan_fwd, l.oracle_scan_fwd_blelloch, l.oracle_scan_bwd, l.oracle_step):
            f.restype = ci
        self._l = l
        self.path = path

    def scan_fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, h0=None,
                 nthreads=None, blelloch=False):
        """Forward selective scan.  u/delta/z [Bsz][Dch][L]; B/C [Bsz][N][L];
        A [Dch][N]; D/delta_bias [Dch]; h0 (optional) [Bsz][Dch][N].
        Returns (out [Bsz][Dch][L], h_last [Bsz][Dch][N])."""
        u = _f64(u)
        Bsz, Dch, L = u.shape
        A = _f64(A)
        N = A.shape[1]
        delta, z = _f64(delta, u.shape), _f64(z, u.shape)
        B, C = _f64(B, (Bsz, N, L)), _f64(C, (Bsz, N, L))
        D, bias, h0 = _f64(D, (Dch,)), _f64(delta_bias, (Dch,)), _f64(h0, (Bsz, Dch, N))
        out = np.empty((Bsz, Dch, L))
        h_last = np.empty((Bsz, Dch, N))
        fn = self._l.oracle_scan_fwd_blelloch if blelloch else self._l.oracle_scan_fwd
        rc = fn(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(bias), int(bool(softplus)),
                Bsz, Dch, L, N, _p(h0), _p(out), _p(h_last), nthreads or default_threads())
        if rc:
            raise RuntimeError(f"oracle scan_fwd failed ({rc})")
        return out, h_last

    def scan_bwd(self, u, delta, A, B, C, D, z, delta_bias, softplus, dy, nthreads=None):
        """Backward of scan_fwd (zero initial state) for the loss sum(dy * out).
        Returns a dict with du, ddelta, dA, dB, dC, dD, dz, ddelta_bias
        (None where the matching input was None)."""
        u = _f64(u)
        Bsz, Dch, L = u.shape
        A = _f64(A)
        N = A.shape[1]
        delta, z, dy = _f64(delta, u.shape), _f64(z, u.shape), _f64(dy, u.shape)
        B, C = _f64(B, (Bsz, N, L)), _f64(C, (Bsz, N, L))
        D, bias = _f64(D, (Dch,)), _f64(delta_bias, (Dch,))
        g = {
            "du": np.empty_like(u), "ddelta": np.empty_like(u), "dA": np.empty((Dch, N)),
            "dB": np.empty((Bsz, N, L)), "dC": np.empty((Bsz, N, L)),
            "dD": np.empty(Dch) if D is not None else None,
            "dz": np.empty_like(u) if z is not None else None,
            "ddelta_bias": np.empty(Dch) if bias is not None else None,
        }
        rc = self._l.oracle_scan_bwd(
            _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(bias), int(bool(softplus)),
            Bsz, Dch, L, N, _p(dy), _p(g["du"]), _p(g["ddelta"]), _p(g["dA"]), _p(g["dB"]),
            _p(g["dC"]), _p(g["dD"]), _p(g["dz"]), _p(g["ddelta_bias"]),
            nthreads or default_threads())
        if rc:
            raise RuntimeError(f"oracle scan_bwd failed ({rc})")
        return g

    def step(self, h, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
             nthreads=None):
        """One-token update.  h [Bsz][Dch][N] is not modified; the new state
        is returned.  u/delta/z [Bsz][Dch]; B/C [Bsz][N].  Returns (y, h_new)."""
        h = np.array(h, dtype=np.float64, copy=True, order="C")
        Bsz, Dch, N = h.shape
        u = _f64(u, (Bsz, Dch))
        delta, z = _f64(delta, (Bsz, Dch)), _f64(z, (Bsz, Dch))
        A, B, C = _f64(A, (Dch, N)), _f64(B, (Bsz, N)), _f64(C, (Bsz, N))
        D, bias = _f64(D, (Dch,)), _f64(delta_bias, (Dch,))
        y = np.empty((Bsz, Dch))
        rc = self._l.oracle_step(_p(h), _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z),
                                 _p(bias), int(bool(softplus)), Bsz, Dch, N, _p(y),
                                 nthreads or default_threads())
        if rc:
            raise RuntimeError(f"oracle step failed ({rc})")
        return y, h


    def conv1d_silu(self, x, w, bias=None, silu=True, nthreads=None):
        """Causal depthwise conv1d (width K) + silu.  x [Bsz][Dch][L], w [Dch][K],
        bias [Dch] or None.  Returns u [Bsz][Dch][L]."""
        x = _f64(x)
        Bsz, Dch, L = x.shape
        w = _f64(w)
        K = w.shape[1]
        bias = _f64(bias, (Dch,))
        u = np.empty_like(x)
        rc = self._l.oracle_conv1d_silu(_p(x), _p(w), _p(bias), int(bool(silu)), Bsz, Dch, L, K,
                                        _p(u), nthreads or default_threads())
        if rc:
            raise RuntimeError(f"oracle conv1d_silu failed ({rc})")
        return u

    def conv1d_silu_bwd(self, x, w, bias, silu, g, nthreads=None):
        """Backward of conv1d_silu for upstream gradient g.  Returns dict dx, dw, dbias
        (dbias None when bias is None)."""
        x = _f64(x)
        Bsz, Dch, L = x.shape
        w = _f64(w)
        K = w.shape[1]
        bias = _f64(bias, (Dch,))
        g = _f64(g, (Bsz, Dch, L))
        out = {"dx": np.empty_like(x), "dw": np.empty((Dch, K)),
               "dbias": np.empty(Dch) if bias is not None else None}
        rc = self._l.oracle_conv1d_silu_bwd(_p(x), _p(w), _p(bias), int(bool(silu)), _p(g), Bsz,
                                            Dch, L, K, _p(out["dx"]), _p(out["dw"]),
                                            _p(out["dbias"]), nthreads or default_threads())
        if rc:
            raise RuntimeError(f"oracle conv1d_silu_bwd failed ({rc})")
        return out

    def xproj(self, u, Wx, Wdt, N, nthreads=None):
        """Input projection (x_proj then dt_proj): u [Bsz][Dch][L], Wx [R+2N][Dch],
        Wdt [Dch][R] -> (delta_raw [Bsz][Dch][L], B [Bsz][N][L], C [Bsz][N][L])."""
        u = _f64(u)
        Bsz, Dch, L = u.shape
        Wdt = _f64(Wdt)
        R = Wdt.shape[1]
        Wx = _f64(Wx, (R + 2 * N, Dch))
        delta = np.zeros((Bsz, Dch, L))
        B = np.zeros((Bsz, N, L))
        C = np.zeros((Bsz, N, L))
        rc = self._l.oracle_xproj(_p(u), _p(Wx), _p(Wdt), Bsz, Dch, L, R, N, _p(delta), _p(B),
                                   _p(C), nthreads or default_threads())
        if rc:
            raise ValueError("oracle_xproj: bad arguments")
        return delta, B, C


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def scan_fwd(*a, **k):
    return default().scan_fwd(*a, **k)


def scan_bwd(*a, **k):
    return default().scan_bwd(*a, **k)


def step(*a, **k):
    return default().step(*a, **k)


def conv1d_silu(*a, **k):
    return default().conv1d_silu(*a, **k)


def conv1d_silu_bwd(*a, **k):
    return default().conv1d_silu_bwd(*a, **k)


def xproj(*a, **k):
    return default().xproj(*a, **k)
