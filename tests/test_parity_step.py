"""Decode step on the GPU (through the C ABI binding) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import check, inputs_to_dev, make_case, oracle_fwd, out_kind, to_dev, to_host64

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu


def _params(dtype, Bsz, Dch, seed):
    cfg = dict(Bsz=Bsz, Dch=Dch, L=1, N=16, dtype=dtype, dt_range=(1e-3, 1e-1), seed=seed)
    return cfg, synth.param_A(Dch, 16), synth.param_D(seed, Dch), \
        synth.param_delta_bias(seed, Dch, cfg["dt_range"])


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch", [(3, 20), (1, 1), (5, 33)])
def test_single_steps(dtype, Bsz, Dch):
    cfg, A, D, bias = _params(dtype, Bsz, Dch, 300 + Dch)
    rng = np.random.default_rng(Dch)
    h0 = rng.standard_normal((Bsz, Dch, 16)).astype(np.float32)
    h = torch.from_numpy(h0).cuda()
    Ad, Dd, bd = (torch.from_numpy(np.array(v)).cuda() for v in (A, D, bias))
    href = h0.astype(np.float64)
    for k in range(4):
        s = synth.step_inputs(cfg, k)
        sd = {n: to_dev(v, dtype) for n, v in s.items()}
        y = ss.ss_step(h, sd["u"], sd["delta"], Ad, sd["B"], sd["C"], Dd, sd["z"], bd, True)
        torch.cuda.synchronize()
        w = {n: synth.widen(v) for n, v in s.items()}
        yref, href = oracle.step(href, w["u"], w["delta"], A, w["B"], w["C"], D, w["z"], bias,
                                 True)
        check(to_host64(y), yref, out_kind(dtype), f"step {k} y")
        check(to_host64(h), href, "f32", f"step {k} h")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_optional_inputs(dtype):
    cfg, A, D, bias = _params(dtype, 2, 24, 5)
    h = torch.zeros((2, 24, 16), device="cuda")
    s = synth.step_inputs(cfg, 0)
    sd = {n: to_dev(v, dtype) for n, v in s.items()}
    y = ss.ss_step(h, sd["u"], sd["delta"], torch.from_numpy(A).cuda(), sd["B"], sd["C"])
    torch.cuda.synchronize()
    w = {n: synth.widen(v) for n, v in s.items()}
    yref, href = oracle.step(np.zeros((2, 24, 16)), w["u"], w["delta"], A, w["B"], w["C"], None,
                             None, None, True)
    check(to_host64(y), yref, out_kind(dtype), "no D/z/bias y")
    check(to_host64(h), href, "f32", "no D/z/bias h")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_scan_then_step_equals_longer_scan(dtype):
    """ss_scan_fwd over L1 steps, its final state handed to ss_step for k more
    tokens == the oracle's scan over L1 + k steps."""
    L1, k = 300, 5
    x = make_case(dtype, 2, 20, L1 + k, seed=31)
    ref, href = oracle_fwd(x)
    head = {n: (v[..., :L1].copy() if n in ("u", "delta", "z", "B", "C") else v)
            for n, v in x.items()}
    xd = inputs_to_dev(head, dtype)
    y, h = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                          xd["delta_bias"], True, return_last_state=True)
    for t in range(L1, L1 + k):
        tok = {n: to_dev(np.ascontiguousarray(x[n][..., t]), dtype)
               for n in ("u", "delta", "z", "B", "C")}
        yt = ss.ss_step(h, tok["u"], tok["delta"], xd["A"], tok["B"], tok["C"], xd["D"], tok["z"],
                        xd["delta_bias"], True)
        torch.cuda.synchronize()
        check(to_host64(yt), ref[..., t], out_kind(dtype), f"token {t}")
    check(to_host64(h), href, "f32", "state after steps")


def test_config4_128_steps_state_checked_every_step():
    """256 x 5120 state, 128 successive bf16 steps from h = 0.  After every
    step, h and y of a 16-batch x 256-channel sub-grid of rows are checked
    against the oracle (rows are independent, so the sub-grid is an exact
    smaller problem), and h of all rows is checked to be finite at the end."""
    cfg = synth.config(4)
    Bsz, Dch = cfg["Bsz"], cfg["Dch"]
    A = synth.param_A(Dch, 16)
    D = synth.param_D(cfg["seed"], Dch)
    bias = synth.param_delta_bias(cfg["seed"], Dch, cfg["dt_range"])
    Ad, Dd, bd = (torch.from_numpy(np.array(v)).cuda() for v in (A, D, bias))
    h = torch.zeros((Bsz, Dch, 16), device="cuda")
    rng = np.random.default_rng(4)
    bsel = np.unique(np.concatenate([[0, Bsz - 1], rng.choice(Bsz, 14, replace=False)]))
    dsel = np.unique(np.concatenate([[0, Dch - 1], rng.choice(Dch, 254, replace=False)]))
    bsel_d, dsel_d = torch.from_numpy(bsel).cuda(), torch.from_numpy(dsel).cuda()
    href = np.zeros((bsel.size, dsel.size, 16))
    for k in range(cfg["steps"]):
        s = synth.step_inputs(cfg, k)
        sd = {n: to_dev(v, "bf16") for n, v in s.items()}
        y = ss.ss_step(h, sd["u"], sd["delta"], Ad, sd["B"], sd["C"], Dd, sd["z"], bd, True)
        w = {n: synth.widen(v) for n, v in s.items()}
        sub = lambda a: a[np.ix_(bsel, dsel)]
        yref, href = oracle.step(href, sub(w["u"]), sub(w["delta"]), A[dsel], w["B"][bsel],
                                 w["C"][bsel], D[dsel], sub(w["z"]), bias[dsel], True)
        torch.cuda.synchronize()
        hs = h.index_select(0, bsel_d).index_select(1, dsel_d)
        ys = y.index_select(0, bsel_d).index_select(1, dsel_d)
        check(to_host64(hs), href, "f32", f"config4 step {k} h")
        check(to_host64(ys), yref, "bf16", f"config4 step {k} y")
    assert torch.isfinite(h).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_steps_back_to_back_without_sync(dtype):
    """Successive steps overlap on the device (each is scheduled while the
    previous runs and waits for it before touching h): 64 steps enqueued with
    no host synchronisation, every token's y kept, then all of them and the
    final state checked against the oracle.  A GPU spin first lets the host
    enqueue every step before the first one runs."""
    Bsz, Dch, steps = 16, 1024, 64
    cfg, A, D, bias = _params(dtype, Bsz, Dch, 404)
    h = torch.zeros((Bsz, Dch, 16), device="cuda")
    Ad, Dd, bd = (torch.from_numpy(np.array(v)).cuda() for v in (A, D, bias))
    toks = [synth.step_inputs(cfg, k) for k in range(steps)]
    dev_toks = [{n: to_dev(v, dtype) for n, v in s.items()} for s in toks]
    ys = [torch.empty((Bsz, Dch), device="cuda", dtype=torch.float32 if dtype == "f32"
                      else torch.bfloat16) for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)
    for k in range(steps):
        sd = dev_toks[k]
        ss.ss_step(h, sd["u"], sd["delta"], Ad, sd["B"], sd["C"], Dd, sd["z"], bd, True, out=ys[k])
    torch.cuda.synchronize()
    href = np.zeros((Bsz, Dch, 16))
    for k in range(steps):
        w = {n: synth.widen(v) for n, v in toks[k].items()}
        yref, href = oracle.step(href, w["u"], w["delta"], A, w["B"], w["C"], D, w["z"], bias, True)
        check(to_host64(ys[k]), yref, out_kind(dtype), f"back-to-back step {k} y")
    check(to_host64(h), href, "f32", "back-to-back final h")
