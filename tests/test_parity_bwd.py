"""Backward scan on the GPU (through the C ABI binding) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (as_io, check, grad_kind, inputs_to_dev, make_case, oracle_bwd, to_dev,
                         to_host64, widen_all)

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

IO_GRADS = ("du", "ddelta", "dz")
F32_GRADS = ("dA", "dB", "dC", "dD", "ddelta_bias")


def run_bwd(xd, dyd, softplus=True, workspace=None):
    return ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd.get("D"),
                          xd.get("z"), xd.get("delta_bias"), softplus, dyd, workspace=workspace)


def compare(x, dtype, softplus=True, what=""):
    dy = x.pop("dy")
    xd = inputs_to_dev(x, dtype)
    g = run_bwd(xd, to_dev(dy, dtype), softplus)
    torch.cuda.synchronize()
    ref = oracle_bwd(x, dy, softplus)
    for k in IO_GRADS + F32_GRADS:
        if ref[k] is None:
            assert g[k] is None, k
            continue
        check(to_host64(g[k]), ref[k], grad_kind(dtype, k in IO_GRADS), f"{what} {k}")


def test_tiny_config_f32():
    cfg = synth.config(0)
    compare(synth.make_inputs(cfg, with_dy=True), "f32", what="tiny")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [
    (3, 20, 1000),
    (1, 16, 256),
    (2, 17, 257),
    (2, 5, 16),
    (1, 3, 1),
    (2, 9, 37),
    (2, 33, 600),
    (2, 3, 2049),   # 17 chunks: the carry walk takes a second block of 16 chunks
    (1, 6, 4500),   # 36 chunks: three blocks, the last one ragged
])
def test_shapes(dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=200 + L + Dch, with_dy=True)
    compare(x, dtype, what=f"{dtype} {Bsz}x{Dch}x{L}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("drop", ["D", "z", "delta_bias", "all", "softplus"])
def test_optional_inputs(dtype, drop):
    x = make_case(dtype, 2, 18, 520, seed=17, with_dy=True)
    softplus = True
    if drop == "all":
        x.update(D=None, z=None, delta_bias=None)
    elif drop == "softplus":
        softplus = False
        d = np.abs(synth.widen(x["delta"])) * 0.05
        x["delta"] = as_io(d, dtype)
        x["delta_bias"] = np.zeros_like(x["delta_bias"])
    else:
        x[drop] = None
    compare(x, dtype, softplus=softplus, what=f"{dtype} drop={drop}")


def test_deterministic_bitwise():
    x = make_case("f32", 3, 40, 1100, seed=21, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "f32")
    dyd = to_dev(dy, "f32")
    g1 = run_bwd(xd, dyd)
    g2 = run_bwd(xd, dyd)
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_workspace_too_small_writes_nothing():
    x = make_case("f32", 2, 16, 300, seed=23, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "f32")
    need = ss.ss_scan_bwd_workspace_size(2, 16, 300)
    small = torch.empty(need - 256, device="cuda", dtype=torch.uint8)
    out = {k: torch.full(s, 5.0, device="cuda") for k, s in
           [("du", (2, 16, 300)), ("ddelta", (2, 16, 300)), ("dA", (16, 16)),
            ("dB", (2, 16, 300)), ("dC", (2, 16, 300)), ("dD", (16,)), ("dz", (2, 16, 300)),
            ("ddelta_bias", (16,))]}
    with pytest.raises(ss.SelscanError) as e:
        ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                       xd["delta_bias"], True, to_dev(dy, "f32"), workspace=small, out=out)
    assert e.value.status == 6
    torch.cuda.synchronize()
    for k, v in out.items():
        assert torch.all(v == 5.0), k


@pytest.mark.parametrize("keep", [True, False])
def test_autograd_wrapper_matches_direct_call(keep):
    """selective_scan's gradients are bitwise those of the direct calls it
    makes: ss_scan_fwd(save_to=ws) + ss_scan_bwd(saved=True) by default,
    ss_scan_bwd alone with keep_chunk_states=False."""
    x = make_case("f32", 2, 16, 300, seed=25, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "f32")
    leaves = {k: v.clone().requires_grad_(True) for k, v in xd.items()}
    y = ss.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                          leaves["D"], leaves["z"], leaves["delta_bias"], True,
                          keep_chunk_states=keep)
    dyd = to_dev(dy, "f32")
    y.backward(dyd)
    if keep:
        ws = torch.empty(ss.ss_scan_bwd_workspace_size(2, 16, 300), device="cuda",
                         dtype=torch.uint8)
        args = (xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                xd["delta_bias"], True)
        ss.ss_scan_fwd(*args, save_to=ws)
        g = ss.ss_scan_bwd(*args, dyd, workspace=ws, saved=True)
    else:
        g = run_bwd(xd, dyd)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
             "delta_bias": "ddelta_bias"}
    for k, gk in names.items():
        assert torch.equal(leaves[k].grad, g[gk]), k


def test_config2_full_size_every_element():
    """8 x 2048 x 2048 float32: every element of all eight gradients against
    the fp64 oracle over the whole workload."""
    cfg = synth.config(2)
    x = synth.make_inputs(cfg, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "f32")
    g = run_bwd(xd, to_dev(dy, "f32"))
    torch.cuda.synchronize()
    ref = oracle_bwd(x, dy, True)
    for k in IO_GRADS + F32_GRADS:
        check(to_host64(g[k]), ref[k], "grad", f"config2 {k}")


def test_stagewise_calls_equal_whole_backward():
    """ss_scan_bwd_states + ss_scan_bwd_reverse + ss_scan_bwd_reduce == ss_scan_bwd, bitwise."""
    x = make_case("bf16", 2, 24, 700, seed=27, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "bf16")
    dyd = to_dev(dy, "bf16")
    g1 = run_bwd(xd, dyd)
    g2 = ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                        xd["delta_bias"], True, dyd,
                        stages=("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce"))
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_empty_backward_zero_gradients():
    dev = "cuda"
    Dch = 4
    A = torch.full((Dch, 16), -1.0, device=dev)
    D = torch.ones(Dch, device=dev)
    bias = torch.zeros(Dch, device=dev)
    u = torch.zeros((2, Dch, 0), device=dev)
    B = torch.zeros((2, 16, 0), device=dev)
    out = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u), "dz": torch.empty_like(u),
           "dA": torch.full((Dch, 16), 9.0, device=dev), "dB": torch.empty_like(B),
           "dC": torch.empty_like(B), "dD": torch.full((Dch,), 9.0, device=dev),
           "ddelta_bias": torch.full((Dch,), 9.0, device=dev)}
    ss.ss_scan_bwd(u, u, A, B, B, D, u, bias, True, u, out=out)
    torch.cuda.synchronize()
    assert torch.all(out["dA"] == 0) and torch.all(out["dD"] == 0)
    assert torch.all(out["ddelta_bias"] == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_softplus_extremes_backward(dtype):
    x = make_case(dtype, 2, 20, 390, seed=33, with_dy=True)
    d = synth.widen(x["delta"]) * 20.0
    x["delta"] = as_io(d, dtype)
    compare(x, dtype, what=f"{dtype} softplus extremes")
