"""Causal depthwise conv1d + silu on the GPU (through the C ABI binding)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check, grad_kind, out_kind, to_dev, to_host64

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

X_ID, W_ID, BIAS_ID, G_ID = 20, 21, 22, 23


def make_conv(dtype, Bsz, Dch, L, K, seed, bias=True):
    x = synth.normal(seed, X_ID, Bsz * Dch * L, dtype).reshape(Bsz, Dch, L)
    w = (synth.normal(seed, W_ID, Dch * K, "f32") / np.sqrt(K)).astype(np.float32).reshape(Dch, K)
    b = synth.normal(seed, BIAS_ID, Dch, "f32") if bias else None
    g = synth.normal(seed, G_ID, Bsz * Dch * L, dtype).reshape(Bsz, Dch, L)
    return x, w, b, g


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("Bsz,Dch,L", [(2, 5, 300), (1, 3, 37), (3, 4, 2), (2, 7, 64)])
def test_forward(dtype, K, Bsz, Dch, L):
    x, w, b, _ = make_conv(dtype, Bsz, Dch, L, K, seed=K * 100 + L)
    u = ss.ss_conv1d_silu(to_dev(x, dtype), dev(w), dev(b), True)
    torch.cuda.synchronize()
    ref = oracle.conv1d_silu(synth.widen(x), w.astype(np.float64), b.astype(np.float64), True)
    check(to_host64(u), ref, out_kind(dtype), f"conv {dtype} K={K} {Bsz}x{Dch}x{L}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_no_bias_no_silu(dtype):
    x, w, _, _ = make_conv(dtype, 2, 6, 120, 4, seed=7, bias=False)
    u = ss.ss_conv1d_silu(to_dev(x, dtype), dev(w), None, False)
    torch.cuda.synchronize()
    ref = oracle.conv1d_silu(synth.widen(x), w.astype(np.float64), None, False)
    check(to_host64(u), ref, out_kind(dtype), "conv no bias, no silu")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("K", [1, 2, 4])
@pytest.mark.parametrize("Bsz,Dch,L", [(2, 5, 300), (1, 3, 37), (3, 4, 3)])
def test_backward(dtype, K, Bsz, Dch, L):
    x, w, b, g = make_conv(dtype, Bsz, Dch, L, K, seed=K * 200 + L)
    out = ss.ss_conv1d_silu_bwd(to_dev(x, dtype), dev(w), dev(b), True, to_dev(g, dtype))
    torch.cuda.synchronize()
    ref = oracle.conv1d_silu_bwd(synth.widen(x), w.astype(np.float64), b.astype(np.float64), True,
                                 synth.widen(g))
    check(to_host64(out["dx"]), ref["dx"], grad_kind(dtype, True), f"conv bwd {dtype} dx")
    check(to_host64(out["dw"]), ref["dw"], "grad", f"conv bwd {dtype} dw")
    check(to_host64(out["dbias"]), ref["dbias"], "grad", f"conv bwd {dtype} dbias")


def test_backward_no_bias_no_silu_and_deterministic():
    x, w, _, g = make_conv("f32", 3, 9, 1000, 4, seed=9, bias=False)
    xd, wd, gd = to_dev(x, "f32"), dev(w), to_dev(g, "f32")
    o1 = ss.ss_conv1d_silu_bwd(xd, wd, None, False, gd)
    o2 = ss.ss_conv1d_silu_bwd(xd, wd, None, False, gd)
    torch.cuda.synchronize()
    assert o1["dbias"] is None
    assert torch.equal(o1["dx"], o2["dx"]) and torch.equal(o1["dw"], o2["dw"])
    ref = oracle.conv1d_silu_bwd(x.astype(np.float64), w.astype(np.float64), None, False,
                                 g.astype(np.float64))
    check(to_host64(o1["dx"]), ref["dx"], "grad", "conv bwd plain dx")
    check(to_host64(o1["dw"]), ref["dw"], "grad", "conv bwd plain dw")


def test_full_size_layer_sampled():
    """8 x 1536 x 2048 bf16 (the Mamba-130M-shaped layer), K = 4: sampled rows
    of u and dx, dw / dbias of sampled channels (all batches)."""
    Bsz, Dch, L, K = 8, 1536, 2048, 4
    x, w, b, g = make_conv("bf16", Bsz, Dch, L, K, seed=1001)
    xd, gd = to_dev(x, "bf16"), to_dev(g, "bf16")
    u = ss.ss_conv1d_silu(xd, dev(w), dev(b), True)
    out = ss.ss_conv1d_silu_bwd(xd, dev(w), dev(b), True, gd)
    torch.cuda.synchronize()
    w64, b64 = w.astype(np.float64), b.astype(np.float64)
    rng = np.random.default_rng(5)
    for d in [0, Dch - 1] + [int(v) for v in rng.integers(Dch, size=6)]:
        sl = slice(d, d + 1)
        xw = synth.widen(x[:, sl])
        ref = oracle.conv1d_silu(xw, w64[sl], b64[sl], True)
        check(to_host64(u[:, sl]), ref, "bf16", f"full-size u channel {d}")
        rb = oracle.conv1d_silu_bwd(xw, w64[sl], b64[sl], True, synth.widen(g[:, sl]))
        check(to_host64(out["dx"][:, sl]), rb["dx"], "bf16", f"full-size dx channel {d}")
        check(to_host64(out["dw"][sl]), rb["dw"], "grad", f"full-size dw channel {d}")
        check(to_host64(out["dbias"][sl]), rb["dbias"], "grad", f"full-size dbias channel {d}")


def test_empty_sequence_zero_parameter_gradients():
    x = torch.zeros((2, 4, 0), device="cuda")
    w = torch.ones((4, 4), device="cuda")
    b = torch.ones(4, device="cuda")
    out = {"dx": torch.empty_like(x), "dw": torch.full((4, 4), 9.0, device="cuda"),
           "dbias": torch.full((4,), 9.0, device="cuda")}
    ss.ss_conv1d_silu_bwd(x, w, b, True, x, out=out)
    torch.cuda.synchronize()
    assert torch.all(out["dw"] == 0) and torch.all(out["dbias"] == 0)
