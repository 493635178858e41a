"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` binding and raises AssertionError
when the oracle disagrees with an independent statement of what the
selective scan computes:

* a brute-force closed form of the scan (products of decays, no recurrence);
* scipy.signal.lfilter for the time-invariant special case (a textbook IIR
  filter), numpy's logaddexp for the softplus discretisation;
* invariants: zero step => zero state, constant inputs => geometric series,
  the gate multiplies after the D skip, scan then step == longer scan,
  a scan resumed from its own final state == the full scan;
* the Blelloch-ordered evaluation of the same scan;
* central finite differences of the forward for every gradient.

The same pins run against mutated builds of oracle.c (tests/test_oracle_mutants.py)
to show that a dropped term, a wrong sign, index or operand fails at least one.
"""
from __future__ import annotations

import numpy as np
from scipy.signal import lfilter
from scipy.special import expit


def _rand_case(rng, Bsz=2, Dch=3, L=20, N=4, dt_lo=1e-2, dt_hi=3e-1):
    u = rng.standard_normal((Bsz, Dch, L))
    delta = rng.standard_normal((Bsz, Dch, L))
    z = rng.standard_normal((Bsz, Dch, L))
    B = rng.standard_normal((Bsz, N, L))
    C = rng.standard_normal((Bsz, N, L))
    A = -(np.arange(N) + 1.0)[None, :] * rng.uniform(0.5, 1.5, size=(Dch, N))
    D = rng.standard_normal(Dch)
    dt = np.exp(rng.uniform(np.log(dt_lo), np.log(dt_hi), size=Dch))
    bias = np.log(np.expm1(dt))
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias)


def _close(got, want, rtol, atol, what):
    got, want = np.asarray(got), np.asarray(want)
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tol; worst at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def brute_force_out(x, softplus=True):
    """y_t = sum_{s<=t} sum_n C_t[n] (prod_{r=s+1..t} a_r[n]) b_s[n] + D u_t,
    then out = y * z * sigmoid(z); a = exp(delta A), b = delta B u."""
    u, A, B, C = x["u"], x["A"], x["B"], x["C"]
    Bsz, Dch, L = u.shape
    raw = x["delta"] + x["delta_bias"][None, :, None]
    dlt = np.logaddexp(0.0, raw) if softplus else raw
    out = np.zeros_like(u)
    for b in range(Bsz):
        for d in range(Dch):
            la = dlt[b, d][:, None] * A[d][None, :]          # [L][N] log a_t
            bb = dlt[b, d][:, None] * B[b].T * u[b, d][:, None]
            cum = np.concatenate([np.zeros((1, A.shape[1])), np.cumsum(la, axis=0)])
            for t in range(L):
                # prod_{r=s+1..t} a_r = exp(cum[t+1] - cum[s+1])
                decay = np.exp(cum[t + 1][None, :] - cum[1 : t + 2])   # [s][N]
                out[b, d, t] = np.sum(C[b][:, t][None, :] * decay * bb[: t + 1])
            out[b, d] += x["D"][d] * u[b, d]
    if x.get("z") is not None:
        out = out * x["z"] * expit(x["z"])
    return out


def pin_closed_form(orc, seed=1):
    rng = np.random.default_rng(seed)
    for softplus in (True, False):
        x = _rand_case(rng, Bsz=2, Dch=3, L=24, N=5)
        if not softplus:
            x["delta"] = np.abs(x["delta"]) * 0.1
        got, _ = orc.scan_fwd(**x, softplus=softplus, nthreads=2)
        _close(got, brute_force_out(x, softplus), 1e-11, 1e-12, f"closed form softplus={softplus}")


def pin_delta_zero(orc, seed=2):
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=3, L=17, N=4)
    x["delta"][:] = 0.0
    x["delta_bias"][:] = 0.0
    out, hl = orc.scan_fwd(**x, softplus=False, nthreads=1)
    want = x["D"][None, :, None] * x["u"] * x["z"] * expit(x["z"])
    _close(out, want, 1e-14, 1e-15, "delta=0 output")
    _close(hl, np.zeros_like(hl), 0, 0, "delta=0 state")


def pin_geometric(orc, seed=3):
    """Constant delta, u and B_n over time: h_t = b (1 - a^{t+1}) / (1 - a)."""
    rng = np.random.default_rng(seed)
    Bsz, Dch, L, N = 1, 2, 50, 3
    c_dt, c_u = 0.07, 1.3
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    A = -np.array([[0.5, 1.0, 3.0], [0.2, 2.0, 7.0]])
    x = dict(u=np.full((Bsz, Dch, L), c_u), delta=np.full((Bsz, Dch, L), c_dt), A=A,
             B=np.broadcast_to(Bn[None, :, None], (Bsz, N, L)).copy(),
             C=np.broadcast_to(Cn[None, :, None], (Bsz, N, L)).copy(),
             D=np.zeros(Dch), z=None, delta_bias=np.zeros(Dch))
    out, hl = orc.scan_fwd(**x, softplus=False, nthreads=1)
    for d in range(Dch):
        a = np.exp(c_dt * A[d])
        b = c_dt * Bn * c_u
        t = np.arange(L)[:, None]
        h = b * (1 - a ** (t + 1)) / (1 - a)                     # [L][N]
        _close(hl[0, d], h[-1], 1e-13, 1e-15, "geometric state")
        _close(out[0, d], h @ Cn, 1e-12, 1e-14, "geometric output")


def pin_lfilter(orc, seed=4):
    """Time-invariant rows are IIR filters: y = sum_n C_n lfilter([dt B_n], [1, -a_n], u) + D u."""
    rng = np.random.default_rng(seed)
    Bsz, Dch, L, N = 2, 3, 70, 4
    Bn = rng.standard_normal((Bsz, N))
    Cn = rng.standard_normal((Bsz, N))
    dts = np.exp(rng.uniform(np.log(1e-2), np.log(0.5), size=Dch))
    A = -(np.arange(N) + 1.0)[None, :] * rng.uniform(0.5, 1.5, size=(Dch, N))
    x = dict(u=rng.standard_normal((Bsz, Dch, L)),
             delta=np.broadcast_to(dts[None, :, None], (Bsz, Dch, L)).copy(), A=A,
             B=np.repeat(Bn[:, :, None], L, axis=2), C=np.repeat(Cn[:, :, None], L, axis=2),
             D=rng.standard_normal(Dch), z=None, delta_bias=None)
    out, _ = orc.scan_fwd(**x, softplus=False, nthreads=1)
    for b in range(Bsz):
        for d in range(Dch):
            want = x["D"][d] * x["u"][b, d]
            for n in range(N):
                a = np.exp(dts[d] * A[d, n])
                want = want + Cn[b, n] * lfilter([dts[d] * Bn[b, n]], [1.0, -a], x["u"][b, d])
            _close(out[b, d], want, 1e-12, 1e-13, "lfilter")


def pin_softplus_cumsum(orc, seed=5):
    """A = 0, B = C = u = 1, D = 0: out_t = sum_{s<=t} softplus(delta_raw_s + bias)."""
    rng = np.random.default_rng(seed)
    Bsz, Dch, L = 2, 3, 40
    raw = rng.standard_normal((Bsz, Dch, L)) * 8.0
    bias = rng.standard_normal(Dch)
    x = dict(u=np.ones((Bsz, Dch, L)), delta=raw, A=np.zeros((Dch, 1)),
             B=np.ones((Bsz, 1, L)), C=np.ones((Bsz, 1, L)), D=np.zeros(Dch), z=None,
             delta_bias=bias)
    out, _ = orc.scan_fwd(**x, softplus=True, nthreads=1)
    want = np.cumsum(np.logaddexp(0.0, raw + bias[None, :, None]), axis=2)
    _close(out, want, 1e-13, 1e-14, "softplus cumsum")
    out, _ = orc.scan_fwd(**x, softplus=False, nthreads=1)
    _close(out, np.cumsum(raw + bias[None, :, None], axis=2), 1e-13, 1e-13, "raw cumsum")


def pin_gate_order(orc, seed=6):
    """The silu gate multiplies the output after the D skip: out = (C h + D u) silu(z)."""
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=4, L=30, N=3)
    gated, _ = orc.scan_fwd(**x, softplus=True, nthreads=1)
    z = x.pop("z")
    plain, _ = orc.scan_fwd(**x, z=None, softplus=True, nthreads=1)
    _close(gated, plain * z * expit(z), 1e-14, 1e-15, "gate order")
    # and the D skip is D_d * u_t
    D = x.pop("D")
    noskip, _ = orc.scan_fwd(**x, D=None, z=None, softplus=True, nthreads=1)
    _close(plain - noskip, D[None, :, None] * x["u"], 1e-13, 1e-13, "D skip")


def pin_blelloch(orc, seed=7):
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=3, L=100, N=6)
    h0 = rng.standard_normal((2, 3, 6))
    a, ha = orc.scan_fwd(**x, softplus=True, h0=h0, nthreads=2)
    b, hb = orc.scan_fwd(**x, softplus=True, h0=h0, nthreads=2, blelloch=True)
    _close(a, b, 1e-12, 1e-13, "blelloch out")
    _close(ha, hb, 1e-12, 1e-13, "blelloch state")


def _slice_t(x, t0, t1):
    y = dict(x)
    for k in ("u", "delta", "z", "B", "C"):
        if y.get(k) is not None:
            y[k] = np.ascontiguousarray(x[k][..., t0:t1])
    return y


def pin_resume(orc, seed=8):
    """Scanning [0, L1) then resuming from its final state over [L1, L) == one scan."""
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=3, L=45, N=4)
    full, hfull = orc.scan_fwd(**x, softplus=True, nthreads=1)
    first, h1 = orc.scan_fwd(**_slice_t(x, 0, 19), softplus=True, nthreads=1)
    second, h2 = orc.scan_fwd(**_slice_t(x, 19, 45), softplus=True, h0=h1, nthreads=1)
    _close(np.concatenate([first, second], axis=2), full, 1e-13, 1e-14, "resume out")
    _close(h2, hfull, 1e-13, 1e-14, "resume state")


def pin_scan_then_step(orc, seed=9):
    """scan(L1) followed by k single-token steps == scan(L1 + k)."""
    rng = np.random.default_rng(seed)
    L1, k = 13, 6
    x = _rand_case(rng, Bsz=2, Dch=3, L=L1 + k, N=4)
    full, hfull = orc.scan_fwd(**x, softplus=True, nthreads=1)
    _, h = orc.scan_fwd(**_slice_t(x, 0, L1), softplus=True, nthreads=1)
    for t in range(L1, L1 + k):
        y, h = orc.step(h, x["u"][..., t], x["delta"][..., t], x["A"], x["B"][..., t],
                        x["C"][..., t], x["D"], x["z"][..., t], x["delta_bias"], softplus=True,
                        nthreads=1)
        _close(y, full[..., t], 1e-13, 1e-14, f"step output t={t}")
    _close(h, hfull, 1e-13, 1e-14, "step state")


_GRAD_KEYS = [("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"),
              ("D", "dD"), ("z", "dz"), ("delta_bias", "ddelta_bias")]


def _fd_check(orc, x, softplus, dy, what):
    def loss(xx):
        out, _ = orc.scan_fwd(**xx, softplus=softplus, nthreads=1)
        return float(np.sum(dy * out))

    g = orc.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                     x["delta_bias"], softplus, dy, nthreads=2)
    for key, gkey in _GRAD_KEYS:
        if x.get(key) is None:
            assert g[gkey] is None, f"{what}: {gkey} should be None"
            continue
        base = x[key]
        fd = np.zeros(base.shape)
        for i in np.ndindex(base.shape):
            eps = 1e-6 * max(1.0, abs(base[i]))
            xp = dict(x)
            arr = base.copy()
            arr[i] = base[i] + eps
            xp[key] = arr
            lp = loss(xp)
            arr = base.copy()
            arr[i] = base[i] - eps
            xp[key] = arr
            lm = loss(xp)
            fd[i] = (lp - lm) / (2 * eps)
        scale = np.sqrt(np.mean(fd ** 2)) + 1e-30
        _close(g[gkey], fd, 1e-6, 1e-6 * scale, f"{what}: {gkey} vs finite differences")


def pin_bwd_fd(orc, seed=10):
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=3, L=11, N=4, dt_lo=0.05, dt_hi=0.6)
    dy = rng.standard_normal(x["u"].shape)
    _fd_check(orc, x, True, dy, "bwd full")


def pin_bwd_fd_plain(orc, seed=11):
    rng = np.random.default_rng(seed)
    x = _rand_case(rng, Bsz=2, Dch=2, L=9, N=3)
    x["delta"] = np.abs(x["delta"]) * 0.2
    x.update(D=None, z=None, delta_bias=None)
    dy = rng.standard_normal(x["u"].shape)
    _fd_check(orc, x, False, dy, "bwd plain")


# ---------------------------------------------------------------------------
# causal depthwise conv1d + silu
# ---------------------------------------------------------------------------
def _conv_case(rng, Bsz=2, Dch=3, L=19, K=4):
    return (rng.standard_normal((Bsz, Dch, L)), rng.standard_normal((Dch, K)),
            rng.standard_normal(Dch))


def pin_conv_convolve(orc, seed=12):
    """Each row is numpy's full convolution with the flipped taps, first L
    outputs (left zero padding), plus bias, then x sigmoid(x) (scipy expit)."""
    rng = np.random.default_rng(seed)
    for K in (1, 2, 4):
        x, w, bias = _conv_case(rng, K=K)
        Bsz, Dch, L = x.shape
        want = np.empty_like(x)
        for b in range(Bsz):
            for d in range(Dch):
                want[b, d] = np.convolve(x[b, d], w[d][::-1])[:L] + bias[d]
        _close(orc.conv1d_silu(x, w, bias, silu=False, nthreads=2), want, 1e-13, 1e-14,
               f"conv K={K}")
        _close(orc.conv1d_silu(x, w, bias, silu=True, nthreads=2), want * expit(want), 1e-13,
               1e-14, f"conv+silu K={K}")


def pin_conv_lfilter(orc, seed=13):
    """The causal convolution is the FIR filter lfilter(w reversed, [1], x)."""
    rng = np.random.default_rng(seed)
    x, w, _ = _conv_case(rng, Bsz=1, Dch=4, L=33, K=4)
    got = orc.conv1d_silu(x, w, None, silu=False, nthreads=1)
    for d in range(4):
        _close(got[0, d], lfilter(w[d][::-1], [1.0], x[0, d]), 1e-13, 1e-14, "conv lfilter")


def pin_conv_impulse(orc, seed=14):
    """A unit impulse at t0 returns the taps w[K-1], w[K-2], ..., w[0] at t0 .. t0+K-1."""
    rng = np.random.default_rng(seed)
    K, L, t0 = 4, 12, 3
    w = rng.standard_normal((1, K))
    x = np.zeros((1, 1, L))
    x[0, 0, t0] = 1.0
    got = orc.conv1d_silu(x, w, None, silu=False, nthreads=1)[0, 0]
    want = np.zeros(L)
    want[t0:t0 + K] = w[0][::-1]
    _close(got, want, 0, 1e-15, "conv impulse")


def pin_conv_bwd_fd(orc, seed=15):
    """Central differences of sum(g * u) for x, w and bias."""
    rng = np.random.default_rng(seed)
    x, w, bias = _conv_case(rng, Bsz=2, Dch=2, L=9, K=4)
    g = rng.standard_normal(x.shape)
    got = orc.conv1d_silu_bwd(x, w, bias, True, g, nthreads=1)
    loss = lambda xx, ww, bb: float(np.sum(g * orc.conv1d_silu(xx, ww, bb, True, nthreads=1)))
    eps = 1e-6
    for name, arr in (("dx", x), ("dw", w), ("dbias", bias)):
        num = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[i] += eps
            lo[i] -= eps
            args_hi = {"dx": (hi, w, bias), "dw": (x, hi, bias), "dbias": (x, w, hi)}[name]
            args_lo = {"dx": (lo, w, bias), "dw": (x, lo, bias), "dbias": (x, w, lo)}[name]
            num[i] = (loss(*args_hi) - loss(*args_lo)) / (2 * eps)
        _close(got[name], num, 1e-6, 1e-7, f"conv finite differences {name}")


def pin_xproj_one_hot(orc, seed=16):
    """One-hot projection weights pick channels: every output is a copy of one
    input channel (pins which weight index is the feature and which the
    channel, the split of xdbl into the dt part, B and C, and the dt_proj
    contraction index)."""
    rng = np.random.default_rng(seed)
    Bsz, Dch, L, R, N = 2, 7, 5, 2, 3
    M = R + 2 * N
    u = rng.standard_normal((Bsz, Dch, L))
    pick = rng.integers(Dch, size=M)          # feature m <- channel pick[m]
    Wx = np.zeros((M, Dch))
    Wx[np.arange(M), pick] = 1.0
    via = rng.integers(R, size=Dch)           # delta channel d <- dt feature via[d]
    Wdt = np.zeros((Dch, R))
    Wdt[np.arange(Dch), via] = 1.0
    delta, B, C = orc.xproj(u, Wx, Wdt, N, nthreads=1)
    _close(delta, u[:, pick[via], :], 0, 0, "xproj one-hot delta")
    _close(B, u[:, pick[R:R + N], :], 0, 0, "xproj one-hot B")
    _close(C, u[:, pick[R + N:], :], 0, 0, "xproj one-hot C")


def pin_xproj_merged_weights(orc, seed=17):
    """The pages' observation: with no bias in x_proj, x_proj then dt_proj is
    one projection by the merged weight Wdt Wx[:R] (numpy matmuls in the
    merged association order)."""
    rng = np.random.default_rng(seed)
    Bsz, Dch, L, R, N = 2, 12, 9, 4, 3
    u = rng.standard_normal((Bsz, Dch, L))
    Wx = rng.standard_normal((R + 2 * N, Dch))
    Wdt = rng.standard_normal((Dch, R))
    delta, B, C = orc.xproj(u, Wx, Wdt, N, nthreads=2)
    merged = Wdt @ Wx[:R]
    _close(delta, np.matmul(merged, u), 0, 1e-12, "xproj merged delta")
    _close(B, np.matmul(Wx[R:R + N], u), 0, 1e-12, "xproj B")
    _close(C, np.matmul(Wx[R + N:], u), 0, 1e-12, "xproj C")


ALL_PINS = [pin_closed_form, pin_delta_zero, pin_geometric, pin_lfilter, pin_softplus_cumsum,
            pin_gate_order, pin_blelloch, pin_resume, pin_scan_then_step, pin_bwd_fd,
            pin_bwd_fd_plain, pin_conv_convolve, pin_conv_lfilter, pin_conv_impulse,
            pin_conv_bwd_fd, pin_xproj_one_hot, pin_xproj_merged_weights]
