"""Helpers for the GPU-vs-oracle parity tests: tolerances, host<->device
conversion of the generator's arrays, and oracle calls on exactly the
values the GPU consumed (bf16 inputs are widened exactly to float64)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Tolerances (the floating-point bars of the parity tests).
#  float32 I/O:                 |err| <= 1e-4 + 1e-4 |ref|
#  bf16 I/O, fp32 accumulation: |err| <= 2e-2 (|ref| + 1e-2), oracle on the same bf16 inputs
#  fp16 I/O, fp32 accumulation: |err| <= 2.5e-3 (|ref| + 1e-2): the bf16 bound scaled by the
#    ratio of the two formats' unit roundoffs (2^-11 against 2^-8, about 5x the roundoff each)
#  gradients kept in float32:   |err| <= 1e-3 (|ref| + rms(ref))
#  gradients stored in bf16 use the bf16 bound (their own rounding is 2^-9 relative).
F32_ATOL, F32_RTOL = 1e-4, 1e-4
BF16_REL, BF16_FLOOR = 2e-2, 1e-2
F16_REL, F16_FLOOR = 2.5e-3, 1e-2
GRAD_REL = 1e-3


def to_dev(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Generator array (float32, float16, or uint16 bf16 bits) -> CUDA tensor of the I/O dtype."""
    if dtype == "bf16":
        assert a.dtype == np.uint16
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)
    if dtype == "f16":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def as_io(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float values to the I/O dtype's host representation."""
    if dtype == "bf16":
        return synth.to_bf16(np.asarray(a, dtype=np.float32))
    if dtype == "f16":
        return synth.to_f16(a)
    return np.asarray(a, dtype=np.float32)


def to_host64(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> exact float64 numpy copy."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def inputs_to_dev(x: dict, dtype: str) -> dict:
    out = {}
    for k, v in x.items():
        if v is None:
            out[k] = None
        elif k in ("A", "D", "delta_bias"):
            out[k] = torch.from_numpy(np.array(v, dtype=np.float32)).cuda()
        else:
            out[k] = to_dev(v, dtype)
    return out


def widen_all(x: dict) -> dict:
    return {k: (None if v is None else synth.widen(v)) for k, v in x.items()}


def check(got, ref, kind: str, what: str):
    """Element-wise tolerance check; kind in {'f32', 'bf16', 'grad'}."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    if kind == "f32":
        bound = F32_ATOL + F32_RTOL * np.abs(ref)
    elif kind == "bf16":
        bound = BF16_REL * (np.abs(ref) + BF16_FLOOR)
    elif kind == "f16":
        bound = F16_REL * (np.abs(ref) + F16_FLOOR)
    elif kind == "grad":
        rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
        bound = GRAD_REL * (np.abs(ref) + rms)
    else:
        raise ValueError(kind)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)
        raise AssertionError(
            f"{what} [{kind}]: {int(bad.sum())}/{err.size} out of tolerance; worst at {i}: "
            f"got {got[i]:.9g} ref {ref[i]:.9g} err {err[i]:.3g} bound {bound[i]:.3g}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0


def out_kind(dtype: str) -> str:
    return dtype if dtype in ("bf16", "f16") else "f32"


def grad_kind(dtype: str, stored_in_io: bool) -> str:
    return dtype if (dtype in ("bf16", "f16") and stored_in_io) else "grad"


def oracle_fwd(x: dict, softplus=True, h0=None):
    w = widen_all(x)
    return oracle.scan_fwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w.get("D"), w.get("z"),
                           w.get("delta_bias"), softplus, h0=h0)


def oracle_bwd(x: dict, dy: np.ndarray, softplus=True):
    w = widen_all(x)
    return oracle.scan_bwd(w["u"], w["delta"], w["A"], w["B"], w["C"], w.get("D"), w.get("z"),
                           w.get("delta_bias"), softplus, synth.widen(dy))


def make_case(dtype: str, Bsz: int, Dch: int, L: int, seed: int, dt_range=(1e-3, 1e-1),
              with_dy=False, N=16):
    cfg = dict(Bsz=Bsz, Dch=Dch, L=L, N=N, dtype=dtype, dt_range=dt_range, seed=seed)
    return synth.make_inputs(cfg, with_dy=with_dy)
