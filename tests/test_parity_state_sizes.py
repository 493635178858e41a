"""State sizes other than 16 (d_state = 8, 32, 64) on the GPU against the
fp64 oracle: the forward scans (the row-sequential kernel, 16-byte and
element-wise rows), the backward (the chunk-parallel kernels with state
groups) and the one-token step."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (as_io, check, grad_kind, inputs_to_dev, make_case, oracle_bwd, oracle_fwd,
                         out_kind, to_dev, to_host64)

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

NS = [8, 32, 64]


def h_kind(dtype):
    # the state is float32 whatever the I/O type; the oracle runs on the same
    # rounded inputs, so h takes the fp32 bar
    return "f32"


@pytest.mark.parametrize("N", NS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [
    (2, 20, 296),   # 16-byte rows in every dtype; channels not a multiple of the CTA
    (3, 40, 300),   # 16-byte rows for fp32 only: element-wise path for 16-bit I/O
    (1, 33, 37),    # element-wise rows, ragged tile
    (2, 5, 1),      # a single step
])
def test_forward(N, dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=500 + N + L, N=N)
    xd = inputs_to_dev(x, dtype)
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x)
    check(to_host64(y), ref, out_kind(dtype), f"N={N} {dtype} {Bsz}x{Dch}x{L} y")
    check(to_host64(hl), href, h_kind(dtype), f"N={N} {dtype} h_last")


@pytest.mark.parametrize("N", NS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_optional_inputs_and_no_softplus(N, dtype):
    x = make_case(dtype, 2, 36, 160, seed=77 + N, N=N)
    x.update(D=None, z=None)
    # without softplus the raw deltas are the steps: keep them positive and small
    x["delta"] = as_io(np.abs(synth.widen(x["delta"])) * 0.05, dtype)
    x["delta_bias"] = np.zeros_like(x["delta_bias"])
    xd = inputs_to_dev(x, dtype)
    y = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], None, None,
                       xd["delta_bias"], False)
    torch.cuda.synchronize()
    ref, _ = oracle_fwd(x, softplus=False)
    check(to_host64(y), ref, out_kind(dtype), f"N={N} {dtype} no D, z, softplus")


@pytest.mark.parametrize("N", NS)
def test_forward_many_rows(N):
    """8192 rows or more: the same kernel as with few rows for N != 16."""
    x = make_case("bf16", 4, 2050, 40, seed=90 + N, N=N)
    xd = inputs_to_dev(x, "bf16")
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x)
    check(to_host64(y), ref, "bf16", f"N={N} many rows y")
    check(to_host64(hl), href, "f32", f"N={N} many rows h_last")


@pytest.mark.parametrize("N", NS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_from_state_in_place(N, dtype):
    Bsz, Dch, L = 2, 24, 120
    x = make_case(dtype, Bsz, Dch, L, seed=40 + N, N=N)
    h0 = np.random.default_rng(N).standard_normal((Bsz, Dch, N)).astype(np.float32)
    xd = inputs_to_dev(x, dtype)
    h = torch.from_numpy(h0).cuda()
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True, h0=h, h_last=h)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x, True, h0=h0.astype(np.float64))
    check(to_host64(y), ref, out_kind(dtype), f"N={N} from state y")
    check(to_host64(hl), href, h_kind(dtype), f"N={N} from state h_last")


@pytest.mark.parametrize("N", NS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch", [(3, 20), (2, 65)])
def test_step(N, dtype, Bsz, Dch):
    cfg = dict(Bsz=Bsz, Dch=Dch, L=1, N=N, dtype=dtype, dt_range=(1e-3, 1e-1), seed=60 + N)
    A = synth.param_A(Dch, N)
    D = synth.param_D(cfg["seed"], Dch)
    bias = synth.param_delta_bias(cfg["seed"], Dch, cfg["dt_range"])
    h0 = np.random.default_rng(Dch + N).standard_normal((Bsz, Dch, N)).astype(np.float32)
    h = torch.from_numpy(h0).cuda()
    Ad, Dd, bd = (torch.from_numpy(np.array(v)).cuda() for v in (A, D, bias))
    href = h0.astype(np.float64)
    for k in range(3):
        s = synth.step_inputs(cfg, k)
        sd = {n: to_dev(v, dtype) for n, v in s.items()}
        y = ss.ss_step(h, sd["u"], sd["delta"], Ad, sd["B"], sd["C"], Dd, sd["z"], bd, True)
        torch.cuda.synchronize()
        w = {n: synth.widen(v) for n, v in s.items()}
        yref, href = oracle.step(href, w["u"], w["delta"], A, w["B"], w["C"], D, w["z"], bias,
                                 True)
        check(to_host64(y), yref, out_kind(dtype), f"N={N} step {k} y")
        check(to_host64(h), href, "f32", f"N={N} step {k} h")


@pytest.mark.parametrize("N", NS)
def test_scan_then_step_equals_longer_scan(N):
    L1, k = 96, 3
    x = make_case("bf16", 2, 20, L1 + k, seed=31 + N, N=N)
    ref, href = oracle_fwd(x)
    head = {n: (v[..., :L1].copy() if n in ("u", "delta", "z", "B", "C") else v)
            for n, v in x.items()}
    xd = inputs_to_dev(head, "bf16")
    _, h = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                          xd["delta_bias"], True, return_last_state=True)
    for t in range(L1, L1 + k):
        tok = {n: to_dev(np.ascontiguousarray(x[n][..., t]), "bf16")
               for n in ("u", "delta", "z", "B", "C")}
        yt = ss.ss_step(h, tok["u"], tok["delta"], xd["A"], tok["B"], tok["C"], xd["D"], tok["z"],
                        xd["delta_bias"], True)
        torch.cuda.synchronize()
        check(to_host64(yt), ref[..., t], "bf16", f"N={N} token {t}")
    check(to_host64(h), href, "f32", f"N={N} state after steps")


IO_GRADS = ("du", "ddelta", "dz")
F32_GRADS = ("dA", "dB", "dC", "dD", "ddelta_bias")


def compare_bwd(x, dtype, what, softplus=True):
    dy = x.pop("dy")
    xd = inputs_to_dev(x, dtype)
    g = ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd.get("D"), xd.get("z"),
                       xd.get("delta_bias"), softplus, to_dev(dy, dtype))
    torch.cuda.synchronize()
    ref = oracle_bwd(x, dy, softplus)
    for k in IO_GRADS + F32_GRADS:
        if ref[k] is None:
            assert g[k] is None, k
            continue
        check(to_host64(g[k]), ref[k], grad_kind(dtype, k in IO_GRADS), f"{what} {k}")


@pytest.mark.parametrize("N", NS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [
    (2, 20, 300),   # several 128-step chunks, a ragged last chunk
    (1, 130, 136),  # two 128-row blocks, element-wise rows for 16-bit I/O
    (2, 9, 37),     # element-wise rows
])
def test_backward(N, dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=700 + N + L, with_dy=True, N=N)
    compare_bwd(x, dtype, f"N={N} {dtype} {Bsz}x{Dch}x{L}")


@pytest.mark.parametrize("N", NS)
def test_backward_optional_inputs_and_no_softplus(N):
    x = make_case("f32", 2, 18, 200, seed=80 + N, with_dy=True, N=N)
    x.update(D=None, z=None, delta_bias=None)
    x["delta"] = as_io(np.abs(synth.widen(x["delta"])) * 0.05, "f32")
    compare_bwd(x, "f32", f"N={N} no D, z, bias, softplus", softplus=False)


@pytest.mark.parametrize("N", NS)
def test_backward_deterministic(N):
    x = make_case("bf16", 2, 40, 400, seed=5, with_dy=True, N=N)
    dy = to_dev(x.pop("dy"), "bf16")
    xd = inputs_to_dev(x, "bf16")
    args = (xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"], xd["delta_bias"],
            True, dy)
    g1, g2 = ss.ss_scan_bwd(*args), ss.ss_scan_bwd(*args)
    torch.cuda.synchronize()
    for k, v in g1.items():
        assert torch.equal(v, g2[k]), k
