"""libselscan: the selective scan of the Mamba selective SSM on NVIDIA B300.

Python binding of the C ABI in ``include/selscan.h``.  This module only
marshals arguments (PyTorch supplies device memory and streams); every step
of the computation runs in the CUDA kernels of ``libselscan.so``.  There is
no CPU or PyTorch fallback: importing fails loudly when the library is
missing or cannot be loaded.

Entry points (same names as the C ABI):
    ss_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                return_last_state=False) -> y | (y, h_last)
    ss_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dy) -> dict of grads
    ss_step(h, u_t, delta_t, A, B_t, C_t, D=None, z_t=None, delta_bias=None,
            softplus=True) -> y_t          (h updated in place)
    ss_scan_bwd_workspace_size(Bsz, Dch, L, N, dtype) -> bytes
and the autograd wrapper ``selective_scan`` (SelectiveScanFn).

Layouts (channel-major, time innermost): u, delta, z, y: (Bsz, Dch, L);
B, C: (Bsz, N, L); A: (Dch, N) float32; D, delta_bias: (Dch,) float32;
h: (Bsz, Dch, N) float32.  N is 8, 16, 32 or 64 (16 is the tuned size).  A
model holding activations as (B, L, D) (the
"mamba.py" page's module boundary) transposes to (B, D, L) before the scan.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libselscan.so")

SS_F32, SS_BF16, SS_F16 = 0, 1, 2
SS_OK, SS_ERR_TIMEOUT = 0, 9
N_STATE = 16


class SelscanError(RuntimeError):
    """A libselscan call returned a non-zero ss_status."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libselscan.so not found at {LIB_PATH}; build it with "
            "`python selective_state_space_114_b300/build.py` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.ss_status_str.argtypes = [ci]
    lib.ss_status_str.restype = ctypes.c_char_p
    lib.ss_version.argtypes = []
    lib.ss_version.restype = ci
    lib.ss_scan_fwd.argtypes = [p] * 8 + [ci, i64, i64, i64, i64, ci, p, p, p]
    lib.ss_scan_fwd.restype = ci
    lib.ss_scan_fwd_from_state.argtypes = [p] * 8 + [ci, p, i64, i64, i64, i64, ci, p, p, p]
    lib.ss_scan_fwd_from_state.restype = ci
    lib.ss_scan_fwd_save.argtypes = [p] * 8 + [ci, i64, i64, i64, i64, ci, p, p, p, sz, p]
    lib.ss_scan_fwd_save.restype = ci
    lib.ss_scan_bwd_workspace_size.argtypes = [i64, i64, i64, i64, ci, ctypes.POINTER(sz)]
    lib.ss_scan_bwd_workspace_size.restype = ci
    lib.ss_scan_bwd.argtypes = ([p] * 8 + [ci, p, i64, i64, i64, i64, ci] + [p] * 8 +
                                [p, sz, p])
    lib.ss_scan_bwd.restype = ci
    for name in ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce",
                 "ss_scan_bwd_saved", "ss_scan_bwd_states_saved"):
        f = getattr(lib, name)
        f.argtypes = lib.ss_scan_bwd.argtypes
        f.restype = ci
    lib.ss_step.argtypes = [p] * 9 + [ci, i64, i64, i64, ci, p, p]
    lib.ss_step.restype = ci
    lib.ss_xproj.argtypes = [p] * 3 + [i64] * 5 + [ci] + [p] * 4
    lib.ss_xproj.restype = ci
    lib.ss_xproj_wait_failures.argtypes = []
    lib.ss_xproj_wait_failures.restype = ci
    lib.ss_check_device_errors.argtypes = [p]
    lib.ss_check_device_errors.restype = ci
    lib.ss_debug_xproj_stuck_wait.argtypes = [ci]
    lib.ss_debug_xproj_stuck_wait.restype = None
    lib.ss_conv1d_silu_fwd.argtypes = [p, p, p, ci, i64, i64, i64, i64, ci, p, p]
    lib.ss_conv1d_silu_fwd.restype = ci
    lib.ss_conv1d_silu_bwd.argtypes = [p, p, p, ci, p, i64, i64, i64, i64, ci, p, p, p, p]
    lib.ss_conv1d_silu_bwd.restype = ci
    lib.ss_scan_bwd_noalloc.argtypes = [p] * 8 + [ci, p, i64, i64, i64, i64, ci] + [p] * 9
    lib.ss_scan_bwd_noalloc.restype = ci
    lib.ss_scan_bwd_noalloc_max_scratch.argtypes = []
    lib.ss_scan_bwd_noalloc_max_scratch.restype = sz
    return lib


_lib = _load()
EXPORTED_SYMBOLS = ("ss_status_str", "ss_version", "ss_scan_fwd", "ss_scan_fwd_from_state",
                    "ss_scan_fwd_save", "ss_scan_bwd_workspace_size",
                    "ss_scan_bwd", "ss_scan_bwd_states", "ss_scan_bwd_reverse",
                    "ss_scan_bwd_reduce", "ss_scan_bwd_saved", "ss_scan_bwd_states_saved", "ss_step", "ss_conv1d_silu_fwd",
                    "ss_conv1d_silu_bwd", "ss_scan_bwd_noalloc",
                    "ss_scan_bwd_noalloc_max_scratch", "ss_xproj", "ss_xproj_wait_failures",
                    "ss_check_device_errors", "ss_debug_xproj_stuck_wait")


def lib() -> ctypes.CDLL:
    return _lib


def ss_status_str(status: int) -> str:
    return _lib.ss_status_str(int(status)).decode()


def ss_version() -> int:
    return int(_lib.ss_version())


def _check(fn: str, status: int):
    if status != 0:
        raise SelscanError(fn, status, ss_status_str(status))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SS_F32
    if t.dtype == torch.bfloat16:
        return SS_BF16
    if t.dtype == torch.float16:
        return SS_F16
    raise TypeError(f"I/O dtype must be float32, bfloat16 or float16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libselscan takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libselscan takes contiguous tensors")
    return t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _same(t, shape, dtype, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def _check_scan_inputs(u, delta, A, B, C, D, z, delta_bias):
    Bsz, Dch, L = u.shape
    N = A.shape[1]
    io = u.dtype
    _same(delta, (Bsz, Dch, L), io, "delta")
    if z is not None:
        _same(z, (Bsz, Dch, L), io, "z")
    _same(B, (Bsz, N, L), io, "B")
    _same(C, (Bsz, N, L), io, "C")
    _same(A, (Dch, N), torch.float32, "A")
    if D is not None:
        _same(D, (Dch,), torch.float32, "D")
    if delta_bias is not None:
        _same(delta_bias, (Dch,), torch.float32, "delta_bias")
    return Bsz, Dch, L, N


def ss_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                return_last_state=False, out=None, h_last=None, h0=None, save_to=None):
    """Forward selective scan on the current CUDA stream; returns y (and the
    final state when return_last_state).  ``h0``: float32 [Bsz][Dch][N]
    state to start from (ss_scan_fwd_from_state); ``h_last`` may be ``h0``.
    ``save_to``: a backward workspace (uint8 CUDA tensor) that also receives
    the chunk states (ss_scan_fwd_save), for ss_scan_bwd(..., saved=True)."""
    Bsz, Dch, L, N = _check_scan_inputs(u, delta, A, B, C, D, z, delta_bias)
    y = torch.empty_like(u) if out is None else out
    if return_last_state and h_last is None:
        h_last = torch.empty((Bsz, Dch, N), device=u.device, dtype=torch.float32)
    if save_to is not None:
        if h0 is not None:
            raise ValueError("save_to: the backward covers the zero initial state only")
        st = _lib.ss_scan_fwd_save(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                   _ptr(z), _ptr(delta_bias), int(bool(softplus)), Bsz, Dch, L, N,
                                   _dtype_code(u), _ptr(y), _ptr(h_last), _ptr(save_to),
                                   save_to.numel(), _stream(u.device))
        _check("ss_scan_fwd_save", st)
    elif h0 is None:
        st = _lib.ss_scan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                              _ptr(delta_bias), int(bool(softplus)), Bsz, Dch, L, N,
                              _dtype_code(u), _ptr(y), _ptr(h_last), _stream(u.device))
        _check("ss_scan_fwd", st)
    else:
        _same(h0, (Bsz, Dch, N), torch.float32, "h0")
        st = _lib.ss_scan_fwd_from_state(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                         _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
                                         Bsz, Dch, L, N, _dtype_code(u), _ptr(y), _ptr(h_last),
                                         _stream(u.device))
        _check("ss_scan_fwd_from_state", st)
    return (y, h_last) if return_last_state else y


def ss_scan_bwd_workspace_size(Bsz, Dch, L, N=N_STATE, dtype=SS_F32) -> int:
    n = ctypes.c_size_t(0)
    _check("ss_scan_bwd_workspace_size",
           _lib.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, dtype, ctypes.byref(n)))
    return int(n.value)


def ss_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus, dy, workspace=None, out=None,
                stages=("ss_scan_bwd",), saved=False):
    """Backward of ss_scan_fwd.  Returns dict du, ddelta, dA, dB, dC, dD, dz,
    ddelta_bias (None for absent optional inputs).  ``workspace``: optional
    uint8 CUDA tensor of at least ss_scan_bwd_workspace_size bytes.
    ``stages``: the C entry points to call in order (default the whole
    backward; ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce")
    is equivalent, one stage per call).  ``saved``: the workspace holds the
    chunk states ss_scan_fwd(..., save_to=workspace) wrote for these inputs;
    the whole backward and its first stage then use the _saved entry points."""
    Bsz, Dch, L, N = _check_scan_inputs(u, delta, A, B, C, D, z, delta_bias)
    _same(dy, (Bsz, Dch, L), u.dtype, "dy")
    dev = u.device
    f32 = torch.float32
    g = out if out is not None else {
        "du": torch.empty_like(u), "ddelta": torch.empty_like(u),
        "dA": torch.empty((Dch, N), device=dev, dtype=f32),
        "dB": torch.empty((Bsz, N, L), device=dev, dtype=f32),
        "dC": torch.empty((Bsz, N, L), device=dev, dtype=f32),
        "dD": torch.empty((Dch,), device=dev, dtype=f32) if D is not None else None,
        "dz": torch.empty_like(u) if z is not None else None,
        "ddelta_bias": torch.empty((Dch,), device=dev, dtype=f32) if delta_bias is not None else None,
    }
    need = ss_scan_bwd_workspace_size(Bsz, Dch, L, N, _dtype_code(u))
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=dev, dtype=torch.uint8)
    args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus)), _ptr(dy), Bsz, Dch, L, N, _dtype_code(u), _ptr(g["du"]),
            _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(workspace), workspace.numel(),
            _stream(dev))
    if saved and workspace is None:
        raise ValueError("saved=True needs the workspace ss_scan_fwd saved to")
    for name in stages:
        if name not in ("ss_scan_bwd", "ss_scan_bwd_states", "ss_scan_bwd_reverse",
                        "ss_scan_bwd_reduce"):
            raise ValueError(name)
        if saved and name in ("ss_scan_bwd", "ss_scan_bwd_states"):
            name += "_saved"
        _check(name, getattr(_lib, name)(*args))
    return g


def ss_step(h, u_t, delta_t, A, B_t, C_t, D=None, z_t=None, delta_bias=None, softplus=True,
            out=None):
    """One decode step; h (Bsz, Dch, N) float32 is updated in place.  Returns y_t."""
    Bsz, Dch, N = h.shape
    _same(h, (Bsz, Dch, N), torch.float32, "h")
    io = u_t.dtype
    _same(u_t, (Bsz, Dch), io, "u_t")
    _same(delta_t, (Bsz, Dch), io, "delta_t")
    if z_t is not None:
        _same(z_t, (Bsz, Dch), io, "z_t")
    _same(B_t, (Bsz, N), io, "B_t")
    _same(C_t, (Bsz, N), io, "C_t")
    _same(A, (Dch, N), torch.float32, "A")
    y = torch.empty_like(u_t) if out is None else out
    st = _lib.ss_step(_ptr(h), _ptr(u_t), _ptr(delta_t), _ptr(A), _ptr(B_t), _ptr(C_t), _ptr(D),
                      _ptr(z_t), _ptr(delta_bias), int(bool(softplus)), Bsz, Dch, N,
                      _dtype_code(u_t), _ptr(y), _stream(h.device))
    _check("ss_step", st)
    return y


class SelectiveScanFn(torch.autograd.Function):
    """Autograd wrapper.  keep_chunk_states (default): forward =
    ss_scan_fwd_save into a backward workspace kept until the backward, which
    is ss_scan_bwd_saved (it recomputes every per-step state but not the
    states at the 128-step chunk boundaries).  Otherwise forward =
    ss_scan_fwd and backward = ss_scan_bwd, which keeps only the inputs."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, D, z, delta_bias, softplus, keep_chunk_states=True):
        ctx.softplus = bool(softplus)
        ctx.save_for_backward(u, delta, A, B, C, D, z, delta_bias)
        ctx.ws = None
        if keep_chunk_states and u.numel() > 0:
            Bsz, Dch, L = u.shape
            n = ss_scan_bwd_workspace_size(Bsz, Dch, L, A.shape[1], _dtype_code(u))
            ctx.ws = torch.empty(max(n, 1), device=u.device, dtype=torch.uint8)
        return ss_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, save_to=ctx.ws)

    @staticmethod
    def backward(ctx, dy):
        u, delta, A, B, C, D, z, delta_bias = ctx.saved_tensors
        g = ss_scan_bwd(u, delta, A, B, C, D, z, delta_bias, ctx.softplus, dy.contiguous(),
                        workspace=ctx.ws, saved=ctx.ws is not None)
        ctx.ws = None
        return (g["du"], g["ddelta"], g["dA"], g["dB"].to(B.dtype), g["dC"].to(C.dtype),
                g["dD"], g["dz"], g["ddelta_bias"], None, None)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True,
                   keep_chunk_states=True):
    """Differentiable selective scan (see SelectiveScanFn)."""
    return SelectiveScanFn.apply(u, delta, A, B, C, D, z, delta_bias, softplus, keep_chunk_states)


def ss_conv1d_silu(x, w, bias=None, silu=True, out=None):
    """Causal depthwise conv1d (width w.shape[1], 1..4) + silu on the current
    CUDA stream: x [Bsz][Dch][L] (I/O dtype), w [Dch][K] and bias [Dch] float32.
    Returns u [Bsz][Dch][L]."""
    if x.dim() != 3 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [Bsz][Dch][L] tensor")
    Bsz, Dch, L = x.shape
    if w.dim() != 2 or w.shape[0] != Dch:
        raise ValueError("w must be [Dch][K]")
    K = w.shape[1]
    _same(w, (Dch, K), torch.float32, "w")
    if bias is not None:
        _same(bias, (Dch,), torch.float32, "bias")
    u = torch.empty_like(x) if out is None else out
    _check("ss_conv1d_silu_fwd",
           _lib.ss_conv1d_silu_fwd(_ptr(x), _ptr(w), _ptr(bias), int(bool(silu)), Bsz, Dch, L, K,
                                   _dtype_code(x), _ptr(u), _stream(x.device)))
    return u


def ss_conv1d_silu_bwd(x, w, bias, silu, du, out=None):
    """Backward of ss_conv1d_silu for the upstream gradient du.  Returns dict
    dx, dw, dbias (dbias None when bias is None)."""
    Bsz, Dch, L = x.shape
    K = w.shape[1]
    _same(du, (Bsz, Dch, L), x.dtype, "du")
    g = out if out is not None else {
        "dx": torch.empty_like(x),
        "dw": torch.empty((Dch, K), device=x.device, dtype=torch.float32),
        "dbias": torch.empty((Dch,), device=x.device, dtype=torch.float32)
        if bias is not None else None,
    }
    _check("ss_conv1d_silu_bwd",
           _lib.ss_conv1d_silu_bwd(_ptr(x), _ptr(w), _ptr(bias), int(bool(silu)), _ptr(du), Bsz,
                                   Dch, L, K, _dtype_code(x), _ptr(g["dx"]), _ptr(g["dw"]),
                                   _ptr(g["dbias"]), _stream(x.device)))
    return g


def ss_xproj(u, Wx, Wdt, N, out=None):
    """Input projection (x_proj then dt_proj, on the tensor cores): u
    [Bsz][Dch][L], Wx [R + 2N][Dch], Wdt [Dch][R], all bf16 or all fp16.
    Returns (delta_raw [Bsz][Dch][L], B [Bsz][N][L], C [Bsz][N][L])."""
    Bsz, Dch, L = u.shape
    R = Wdt.shape[1]
    _same(Wx, (R + 2 * N, Dch), u.dtype, "Wx")
    _same(Wdt, (Dch, R), u.dtype, "Wdt")
    if out is None:
        out = (torch.empty_like(u), torch.empty((Bsz, N, L), device=u.device, dtype=u.dtype),
               torch.empty((Bsz, N, L), device=u.device, dtype=u.dtype))
    delta, B, C = out
    _check("ss_xproj", _lib.ss_xproj(_ptr(u), _ptr(Wx), _ptr(Wdt), Bsz, Dch, L, R, N,
                                     _dtype_code(u), _ptr(delta), _ptr(B), _ptr(C),
                                     _stream(u.device)))
    return delta, B, C


def ss_xproj_wait_failures() -> int:
    return int(_lib.ss_xproj_wait_failures())


def ss_check_device_errors(device=None) -> int:
    """Status of the device error word since the last check (SS_OK or
    SS_ERR_TIMEOUT); synchronises the current stream and clears the word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    return int(_lib.ss_check_device_errors(_stream(dev)))


def ss_debug_xproj_stuck_wait(on: bool) -> None:
    """Test hook: make every later ss_xproj CTA give up one bounded wait."""
    _lib.ss_debug_xproj_stuck_wait(1 if on else 0)
