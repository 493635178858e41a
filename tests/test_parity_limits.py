"""Largest batch a launch takes (the batch is a grid dimension of at most
65535 for the scans and the step; conv1d spreads its rows over two grid
dimensions): every entry point at Bsz = 65535 against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (check, grad_kind, inputs_to_dev, make_case, oracle_bwd, oracle_fwd,
                         out_kind, to_dev, to_host64)

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

BMAX = 65535


@pytest.mark.parametrize("dtype,Dch,L", [
    ("bf16", 2, 16),   # 131070 rows: the row-sequential kernel
    ("f32", 1, 5),     # element-wise rows: the chunked element-wise kernel
])
def test_forward_max_batch(dtype, Dch, L):
    x = make_case(dtype, BMAX, Dch, L, seed=90 + L)
    xd = inputs_to_dev(x, dtype)
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x)
    check(to_host64(y), ref, out_kind(dtype), f"max batch {dtype} y")
    check(to_host64(hl), href, "f32" if dtype == "f32" else out_kind(dtype), "max batch h_last")


def test_backward_max_batch():
    x = make_case("f32", BMAX, 1, 8, seed=91, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "f32")
    g = ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                       xd["delta_bias"], True, to_dev(dy, "f32"))
    torch.cuda.synchronize()
    ref = oracle_bwd(x, dy)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        check(to_host64(g[k]), ref[k], grad_kind("f32", False), f"max batch {k}")


def test_step_max_batch():
    Dch, N = 3, 16
    cfg = dict(Bsz=BMAX, Dch=Dch, L=1, N=N, dtype="bf16", dt_range=(1e-3, 1e-1), seed=92)
    A = synth.param_A(Dch, N)
    D = synth.param_D(cfg["seed"], Dch)
    bias = synth.param_delta_bias(cfg["seed"], Dch, cfg["dt_range"])
    h0 = np.random.default_rng(2).standard_normal((BMAX, Dch, N)).astype(np.float32)
    h = torch.from_numpy(h0).cuda()
    s = synth.step_inputs(cfg, 0)
    sd = {n: to_dev(v, "bf16") for n, v in s.items()}
    y = ss.ss_step(h, sd["u"], sd["delta"], torch.from_numpy(A).cuda(), sd["B"], sd["C"],
                   torch.from_numpy(D).cuda(), sd["z"], torch.from_numpy(bias).cuda(), True)
    torch.cuda.synchronize()
    w = {n: synth.widen(v) for n, v in s.items()}
    yref, href = oracle.step(h0.astype(np.float64), w["u"], w["delta"], A, w["B"], w["C"], D,
                             w["z"], bias, True)
    check(to_host64(y), yref, "bf16", "max batch step y")
    check(to_host64(h), href, "f32", "max batch step h")


def test_conv_rows_beyond_one_grid_dimension():
    """65535 x 2 rows: the forward's row index spans two grid dimensions."""
    Bsz, Dch, L, K = BMAX, 2, 24, 4
    x = synth.normal(93, 20, Bsz * Dch * L, "f32").reshape(Bsz, Dch, L)
    w = (synth.normal(93, 21, Dch * K, "f32") / 2.0).reshape(Dch, K)
    b = synth.normal(93, 22, Dch, "f32")
    u = ss.ss_conv1d_silu(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(),
                          torch.from_numpy(b).cuda(), True)
    torch.cuda.synchronize()
    ref = oracle.conv1d_silu(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64),
                             True)
    check(to_host64(u), ref, "f32", "conv rows beyond one grid dimension")
