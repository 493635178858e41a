"""Input projection (x_proj then dt_proj) on the tensor cores against the fp64
oracle.

Tolerances.  B and C are fp32 sums of the 16-bit products rounded once to the
I/O type: the usual bf16 / fp16 bounds.  delta_raw goes through xdbl[:R]
rounded to the I/O type (unit roundoff e = 2^-9 for bf16, 2^-12 for fp16)
before dt_proj, then through its own rounding, so per element
    |delta_gpu - delta| <= 2e (sum_r |Wdt[d][r]| |xdbl_r|) + 2e |delta| + 1e-5
(a factor two over the first-order error of the two roundings; fp32
accumulation adds far less)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check, out_kind, to_dev, to_host64

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

UNIT = {"bf16": 2.0 ** -9, "f16": 2.0 ** -12}


def make(dtype, Bsz, Dch, L, R, N, seed):
    u = synth.normal(seed, 40, Bsz * Dch * L, dtype).reshape(Bsz, Dch, L)
    wx = synth.normal(seed, 41, (R + 2 * N) * Dch, "f32") / np.sqrt(Dch)
    wdt = synth.normal(seed, 42, Dch * R, "f32") / np.sqrt(R)
    Wx = synth.to_bf16(wx) if dtype == "bf16" else synth.to_f16(wx)
    Wdt = synth.to_bf16(wdt) if dtype == "bf16" else synth.to_f16(wdt)
    return u, Wx.reshape(R + 2 * N, Dch), Wdt.reshape(Dch, R)


def check_xproj(u, Wx, Wdt, N, dtype, got, what):
    u64, Wx64, Wdt64 = synth.widen(u), synth.widen(Wx), synth.widen(Wdt)
    R = Wdt.shape[1]
    delta, B, C = oracle.xproj(u64, Wx64, Wdt64, N)
    check(to_host64(got[1]), B, out_kind(dtype), f"{what} B")
    check(to_host64(got[2]), C, out_kind(dtype), f"{what} C")
    # |xdbl[:R]| per token through a second oracle call with identity dt_proj rows
    Dch = Wdt.shape[0]
    eye = np.zeros((Dch, R))
    eye[np.arange(R), np.arange(R)] = 1.0
    xr, _, _ = oracle.xproj(u64, Wx64, eye, N)          # [Bsz][Dch][L], rows < R = xdbl[:R]
    mag = np.einsum("dr,brt->bdt", np.abs(Wdt64), np.abs(xr[:, :R, :]))
    e = UNIT[dtype]
    bound = 2 * e * mag + 2 * e * np.abs(delta) + 1e-5
    g = to_host64(got[0])
    assert np.all(np.isfinite(g)), f"{what} delta: non-finite"
    err = np.abs(g - delta)
    bad = err > bound
    assert not bad.any(), (f"{what} delta: {int(bad.sum())}/{err.size} out of tolerance; worst "
                           f"ratio {float((err / bound).max()):.3g}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L,R,N", [
    (2, 64, 128, 16, 8),     # one tile, one channel chunk
    (2, 200, 136, 48, 16),   # ragged channel chunk and token tile; the Mamba-130M ratio
    (1, 320, 64, 160, 16),   # dt_rank 160 (Mamba-2.8B ratio), R + 2N = 192
    (3, 136, 256, 8, 4),     # smallest dt_rank; three delta steps of 128 channels (ragged)
])
def test_xproj(dtype, Bsz, Dch, L, R, N):
    u, Wx, Wdt = make(dtype, Bsz, Dch, L, R, N, seed=Dch + L + R)
    got = ss.ss_xproj(to_dev(u, dtype), to_dev(Wx, dtype), to_dev(Wdt, dtype), N)
    torch.cuda.synchronize()
    check_xproj(u, Wx, Wdt, N, dtype, got, f"xproj {dtype} {Bsz}x{Dch}x{L} R={R} N={N}")
    assert ss.ss_check_device_errors() == ss.SS_OK  # no bounded wait gave up


def test_xproj_full_size_sampled_tokens():
    """8 x 1536 x 2048 bf16 (the Mamba-130M layer: R = 48, N = 16); every
    output of 24 sampled tokens against the oracle run on those tokens."""
    Bsz, Dch, L, R, N = 8, 1536, 2048, 48, 16
    u, Wx, Wdt = make("bf16", Bsz, Dch, L, R, N, seed=9)
    got = ss.ss_xproj(to_dev(u, "bf16"), to_dev(Wx, "bf16"), to_dev(Wdt, "bf16"), N)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    ts = np.unique(np.concatenate([[0, 127, 128, L - 1], rng.integers(L, size=20)]))
    sub = tuple(g[:, :, ts].contiguous() for g in got)
    check_xproj(np.ascontiguousarray(u[:, :, ts]), Wx, Wdt, N, "bf16", sub, "xproj full size")
    assert ss.ss_check_device_errors() == ss.SS_OK  # no bounded wait gave up


def test_xproj_deterministic_and_empty():
    u, Wx, Wdt = make("bf16", 2, 64, 128, 16, 8, seed=3)
    ud, wxd, wdtd = to_dev(u, "bf16"), to_dev(Wx, "bf16"), to_dev(Wdt, "bf16")
    a = ss.ss_xproj(ud, wxd, wdtd, 8)
    b = ss.ss_xproj(ud, wxd, wdtd, 8)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    e = torch.zeros((2, 64, 0), device="cuda", dtype=torch.bfloat16)
    d, B, C = ss.ss_xproj(e, wxd, wdtd, 8)
    assert d.shape == (2, 64, 0) and B.shape == (2, 8, 0)
