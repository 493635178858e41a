"""Out-of-bounds stores: every output of the backward, the decode step, the
conv1d + silu (both directions) and the input projection is a view into a
larger buffer whose padding holds a canary value; after the call the padding
must be untouched, and the outputs themselves must match the fp64 oracle.
(The forward's guard test sits with the forward parity tests.)  Shapes are
ragged so that the last tile, chunk and vector of every kernel is partial."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (check, grad_kind, inputs_to_dev, make_case, oracle_bwd, out_kind,
                         to_dev, to_host64)
from test_parity_conv import dev, make_conv
from test_parity_xproj import check_xproj, make

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

PAD = 64  # elements of padding on each side (128 or 256 bytes: views stay 16-byte aligned)
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


class Guarded:
    """A tensor of `shape` inside a buffer padded with a canary value."""

    def __init__(self, shape, dtype, canary=-1234.5):
        self.n = int(np.prod(shape))
        self.canary = canary
        self.buf = torch.full((self.n + 2 * PAD,), canary, device="cuda", dtype=dtype)
        self.view = self.buf[PAD:PAD + self.n].view(*shape)

    def intact(self):
        c = torch.tensor(self.canary, dtype=self.buf.dtype, device="cuda")
        return bool(torch.all(self.buf[:PAD] == c)) and bool(torch.all(self.buf[PAD + self.n:] == c))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [(2, 17, 257), (1, 130, 300)])
def test_backward_writes_only_its_outputs(dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=500 + L, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, dtype)
    io, f32 = TDT[dtype], torch.float32
    g = {"du": Guarded((Bsz, Dch, L), io), "ddelta": Guarded((Bsz, Dch, L), io),
         "dz": Guarded((Bsz, Dch, L), io), "dA": Guarded((Dch, 16), f32),
         "dB": Guarded((Bsz, 16, L), f32), "dC": Guarded((Bsz, 16, L), f32),
         "dD": Guarded((Dch,), f32), "ddelta_bias": Guarded((Dch,), f32)}
    ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                   xd["delta_bias"], True, to_dev(dy, dtype), out={k: v.view for k, v in g.items()})
    torch.cuda.synchronize()
    ref = oracle_bwd(x, dy, True)
    for k, v in g.items():
        assert v.intact(), f"{dtype} {k}: a store landed outside the output"
        check(to_host64(v.view), ref[k], grad_kind(dtype, k in ("du", "ddelta", "dz")),
              f"guarded {dtype} {k}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch", [(3, 33), (1, 65)])
def test_step_writes_only_its_outputs(dtype, Bsz, Dch):
    seed = 600 + Dch
    cfg = dict(Bsz=Bsz, Dch=Dch, L=1, N=16, dtype=dtype, dt_range=(1e-3, 1e-1), seed=seed)
    A, D = synth.param_A(Dch, 16), synth.param_D(seed, Dch)
    bias = synth.param_delta_bias(seed, Dch, cfg["dt_range"])
    h0 = np.random.default_rng(seed).standard_normal((Bsz, Dch, 16)).astype(np.float32)
    h = Guarded((Bsz, Dch, 16), torch.float32)
    h.view.copy_(torch.from_numpy(h0))
    y = Guarded((Bsz, Dch), TDT[dtype])
    s = synth.step_inputs(cfg, 0)
    sd = {n: to_dev(v, dtype) for n, v in s.items()}
    Ad, Dd, bd = (torch.from_numpy(np.array(v)).cuda() for v in (A, D, bias))
    ss.ss_step(h.view, sd["u"], sd["delta"], Ad, sd["B"], sd["C"], Dd, sd["z"], bd, True,
               out=y.view)
    torch.cuda.synchronize()
    assert h.intact() and y.intact()
    w = {n: synth.widen(v) for n, v in s.items()}
    yref, href = oracle.step(h0.astype(np.float64), w["u"], w["delta"], A, w["B"], w["C"], D,
                             w["z"], bias, True)
    check(to_host64(y.view), yref, out_kind(dtype), "guarded step y")
    check(to_host64(h.view), href, "f32", "guarded step h")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("K", [1, 4])
def test_conv1d_writes_only_its_outputs(dtype, K):
    Bsz, Dch, L = 2, 7, 301
    x, w, b, gr = make_conv(dtype, Bsz, Dch, L, K, seed=700 + K)
    xt, gt = to_dev(x, dtype), to_dev(gr, dtype)
    u = Guarded((Bsz, Dch, L), TDT[dtype])
    ss.ss_conv1d_silu(xt, dev(w), dev(b), True, out=u.view)
    gd = {"dx": Guarded((Bsz, Dch, L), TDT[dtype]), "dw": Guarded((Dch, K), torch.float32),
          "dbias": Guarded((Dch,), torch.float32)}
    ss.ss_conv1d_silu_bwd(xt, dev(w), dev(b), True, gt, out={k: v.view for k, v in gd.items()})
    torch.cuda.synchronize()
    assert u.intact(), "conv forward"
    for k, v in gd.items():
        assert v.intact(), f"conv backward {k}"
    x64, w64, b64 = synth.widen(x), w.astype(np.float64), b.astype(np.float64)
    check(to_host64(u.view), oracle.conv1d_silu(x64, w64, b64, True), out_kind(dtype),
          "guarded conv u")
    ref = oracle.conv1d_silu_bwd(x64, w64, b64, True, synth.widen(gr))
    check(to_host64(gd["dx"].view), ref["dx"], grad_kind(dtype, True), "guarded conv dx")
    check(to_host64(gd["dw"].view), ref["dw"], "grad", "guarded conv dw")
    check(to_host64(gd["dbias"].view), ref["dbias"], "grad", "guarded conv dbias")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_xproj_writes_only_its_outputs(dtype):
    Bsz, Dch, L, R, N = 2, 200, 136, 48, 16
    u, Wx, Wdt = make(dtype, Bsz, Dch, L, R, N, seed=801)
    io = TDT[dtype]
    out = (Guarded((Bsz, Dch, L), io), Guarded((Bsz, N, L), io), Guarded((Bsz, N, L), io))
    ss.ss_xproj(to_dev(u, dtype), to_dev(Wx, dtype), to_dev(Wdt, dtype), N,
                out=tuple(o.view for o in out))
    torch.cuda.synchronize()
    assert ss.ss_check_device_errors() == ss.SS_OK
    for name, o in zip(("delta", "B", "C"), out):
        assert o.intact(), f"xproj {name}"
    check_xproj(u, Wx, Wdt, N, dtype, tuple(o.view for o in out), f"guarded xproj {dtype}")
