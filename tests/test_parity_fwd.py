"""Forward scan on the GPU (through the C ABI binding) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_util import (as_io, check, inputs_to_dev, make_case, oracle_fwd, out_kind, to_host64,
                         widen_all)

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu


def run_fwd(xd, softplus=True, last=True):
    return ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd.get("D"),
                          xd.get("z"), xd.get("delta_bias"), softplus, return_last_state=last)


def compare(x, dtype, softplus=True, what=""):
    xd = inputs_to_dev(x, dtype)
    y, hl = run_fwd(xd, softplus)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x, softplus)
    check(to_host64(y), ref, out_kind(dtype), f"{what} y")
    check(to_host64(hl), href, "f32", f"{what} h_last")


def test_tiny_config_f32():
    cfg = synth.config(0)
    compare(synth.make_inputs(cfg), "f32", what="tiny")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [
    (3, 20, 1000),   # several chunks + ragged tail, channels not a multiple of the CTA
    (1, 16, 256),    # exactly one chunk
    (2, 17, 257),    # one step past a chunk
    (2, 5, 16),      # one lane segment
    (1, 3, 1),       # a single step
    (2, 9, 37),      # L not a multiple of the vector width (element-wise path)
    (1, 33, 2050),   # ragged at the vector width for f32 only
])
def test_shapes(dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=100 + L + Dch)
    compare(x, dtype, what=f"{dtype} {Bsz}x{Dch}x{L}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("drop", ["D", "z", "delta_bias", "all", "softplus"])
def test_optional_inputs(dtype, drop):
    x = make_case(dtype, 2, 18, 700, seed=7)
    softplus = True
    if drop == "all":
        x.update(D=None, z=None, delta_bias=None)
    elif drop == "softplus":
        softplus = False
        # raw deltas must be positive-ish for a decaying state: use |delta| * 0.05
        d = synth.widen(x["delta"])
        d = np.abs(d) * 0.05
        x["delta"] = as_io(d, dtype)
        x["delta_bias"] = np.zeros_like(x["delta_bias"])
    else:
        x[drop] = None
    compare(x, dtype, softplus=softplus, what=f"{dtype} drop={drop}")


def test_empty_inputs():
    dev = "cuda"
    A = torch.full((4, 16), -1.0, device=dev)
    for Bsz, Dch, L in [(2, 4, 0), (0, 4, 8)]:
        u = torch.zeros((Bsz, Dch, L), device=dev)
        B = torch.zeros((Bsz, 16, L), device=dev)
        y, hl = ss.ss_scan_fwd(u, u, A[:Dch].contiguous(), B, B, return_last_state=True)
        torch.cuda.synchronize()
        assert y.shape == (Bsz, Dch, L)
        assert hl.shape == (Bsz, Dch, 16) and torch.all(hl == 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_no_writes_outside_outputs(dtype):
    """Guard regions around y and h_last must be untouched (bounds of every store)."""
    x = make_case(dtype, 2, 19, 300, seed=9)
    xd = inputs_to_dev(x, dtype)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}.get(dtype, torch.float32)
    pad = 64
    n = 2 * 19 * 300
    ybuf = torch.full((n + 2 * pad,), 7.0, device="cuda", dtype=tdt)
    hbuf = torch.full((2 * 19 * 16 + 2 * pad,), 7.0, device="cuda", dtype=torch.float32)
    y = ybuf[pad : pad + n].view(2, 19, 300)
    hl = hbuf[pad : pad + 2 * 19 * 16].view(2, 19, 16)
    ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                   xd["delta_bias"], True, out=y, h_last=hl, return_last_state=True)
    torch.cuda.synchronize()
    assert torch.all(ybuf[:pad] == 7.0) and torch.all(ybuf[pad + n :] == 7.0)
    assert torch.all(hbuf[:pad] == 7.0) and torch.all(hbuf[pad + 2 * 19 * 16 :] == 7.0)
    ref, _ = oracle_fwd(x)
    check(to_host64(y), ref, out_kind(dtype), "guarded y")


def test_deterministic():
    x = make_case("bf16", 2, 40, 1500, seed=11)
    xd = inputs_to_dev(x, "bf16")
    y1, h1 = run_fwd(xd)
    y2, h2 = run_fwd(xd)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


def _rows_oracle(cfg, rows):
    """fp64 oracle on the (b, d) rows of a workload, regenerated on their own
    (one oracle call per batch over the sampled channels, all host cores)."""
    L, N = cfg["L"], cfg["N"]
    out = {}
    for b in sorted({b for b, _ in rows}):
        ds = [d for bb, d in rows if bb == b]
        rs = [widen_all(synth.row_inputs(cfg, b, d)) for d in ds]
        st = lambda k: np.stack([r[k] for r in rs]).reshape(1, len(ds), L)
        y, hl = oracle.scan_fwd(st("u"), st("delta"), np.stack([r["A"] for r in rs]),
                                rs[0]["B"].reshape(1, N, L), rs[0]["C"].reshape(1, N, L),
                                np.concatenate([r["D"] for r in rs]), st("z"),
                                np.concatenate([r["delta_bias"] for r in rs]), True)
        for i, d in enumerate(ds):
            out[(b, d)] = (y[0, i], hl[0, i])
    return out


def _check_long_rows(got, ref):
    """The error, relative to the bound, must not grow along the sequence."""
    L = got.shape[-1]
    err = np.abs(got - ref) / (2e-2 * (np.abs(ref) + 1e-2))
    per = err[: (L // 4096) * 4096].reshape(-1, 4096).max(axis=1)
    assert per.max() <= 1.0


def test_config1_full_size_every_element():
    """The bf16 Mamba-130M layer (8 x 1536 x 2048): every output and final
    state against the fp64 oracle over the whole workload."""
    cfg = synth.config(1)
    x = synth.make_inputs(cfg)
    xd = inputs_to_dev(x, cfg["dtype"])
    y, hl = run_fwd(xd)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x)
    check(to_host64(y), ref, "bf16", "config 1 y")
    check(to_host64(hl), href, "f32", "config 1 h_last")


def test_config3_full_size_sampled_rows():
    """1 x 5120 x 131072 bf16 (too large for a whole-workload oracle pass):
    64 sampled rows, including both ends, every step of each."""
    cfg = synth.config(3)
    x = synth.make_inputs(cfg)
    xd = inputs_to_dev(x, cfg["dtype"])
    del x
    y, hl = run_fwd(xd)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    rng = np.random.default_rng(3)
    ds = sorted({0, 5119, *[int(v) for v in rng.choice(5120, size=62, replace=False)]})
    rows = [(0, d) for d in ds]
    refs = _rows_oracle(cfg, rows)
    for b, d in rows:
        ref, href = refs[(b, d)]
        got = to_host64(y[b, d])
        check(got, ref, "bf16", f"config 3 row ({b},{d})")
        check(to_host64(hl[b, d]), href, "f32", f"config 3 h_last ({b},{d})")
        _check_long_rows(got, ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_softplus_extremes(dtype):
    """delta_raw spread over about +-60: both branches of the GPU's log1p
    (series below e^-|x| = 1/32, log2 above) and the saturated ends."""
    x = make_case(dtype, 2, 24, 520, seed=31)
    d = synth.widen(x["delta"]) * 20.0
    x["delta"] = as_io(d, dtype)
    compare(x, dtype, what=f"{dtype} softplus extremes")


def test_config2_full_size_forward_every_element():
    """8 x 2048 x 2048 float32 forward (the fp32 kernel configuration): every
    output and final state against the fp64 oracle."""
    cfg = synth.config(2)
    x = synth.make_inputs(cfg)
    xd = inputs_to_dev(x, "f32")
    y, hl = run_fwd(xd)
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x)
    check(to_host64(y), ref, "f32", "config 2 y")
    check(to_host64(hl), href, "f32", "config 2 h_last")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_zero_step_leaves_only_the_gated_skip(dtype):
    """delta = 0 without softplus: every decay is 1 and every input term 0, so
    the state stays 0 and y = D u silu(z) (up to the output rounding)."""
    x = make_case(dtype, 2, 20, 640, seed=35)
    x["delta"] = np.zeros_like(x["delta"])
    x["delta_bias"] = np.zeros_like(x["delta_bias"])
    xd = inputs_to_dev(x, dtype)
    y, hl = run_fwd(xd, softplus=False)
    torch.cuda.synchronize()
    assert torch.all(hl == 0)
    w = widen_all(x)
    z = w["z"]
    want = w["D"][None, :, None] * w["u"] * z / (1.0 + np.exp(-z))
    check(to_host64(y), want, out_kind(dtype), f"{dtype} zero step")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", [(2, 20, 700), (1, 17, 37), (3, 9, 256)])
def test_from_state_matches_oracle(dtype, Bsz, Dch, L):
    """ss_scan_fwd_from_state against the oracle started from the same h0."""
    x = make_case(dtype, Bsz, Dch, L, seed=50 + L)
    h0 = np.random.default_rng(L).standard_normal((Bsz, Dch, 16)).astype(np.float32)
    xd = inputs_to_dev(x, dtype)
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True,
                           h0=torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    ref, href = oracle_fwd(x, True, h0=h0.astype(np.float64))
    check(to_host64(y), ref, out_kind(dtype), f"{dtype} from state y")
    check(to_host64(hl), href, "f32", "from state h_last")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_two_chunks_in_place_equal_one_scan(dtype):
    """Chunked prefill: scan [0, L1), then continue over [L1, L) from the
    carried state updated in place (h_last = h0) == one scan over [0, L)."""
    L1, L = 512, 1200
    x = make_case(dtype, 2, 18, L, seed=61)
    xd = inputs_to_dev(x, dtype)
    part = lambda t, a, b: t[..., a:b].contiguous()
    y1, h = ss.ss_scan_fwd(*(part(xd[k], 0, L1) for k in ("u", "delta")), xd["A"],
                           part(xd["B"], 0, L1), part(xd["C"], 0, L1), xd["D"],
                           part(xd["z"], 0, L1), xd["delta_bias"], True, return_last_state=True)
    y2, h2 = ss.ss_scan_fwd(*(part(xd[k], L1, L) for k in ("u", "delta")), xd["A"],
                            part(xd["B"], L1, L), part(xd["C"], L1, L), xd["D"],
                            part(xd["z"], L1, L), xd["delta_bias"], True,
                            return_last_state=True, h0=h, h_last=h)
    torch.cuda.synchronize()
    assert h2.data_ptr() == h.data_ptr()
    ref, href = oracle_fwd(x, True)
    check(to_host64(torch.cat([y1, y2], dim=-1)), ref, out_kind(dtype), f"{dtype} chunked y")
    check(to_host64(h), href, "f32", "chunked final state")


def test_from_state_empty_sequence_copies_the_state():
    h0 = torch.randn(2, 4, 16, device="cuda")
    A = torch.full((4, 16), -1.0, device="cuda")
    u = torch.zeros((2, 4, 0), device="cuda")
    B = torch.zeros((2, 16, 0), device="cuda")
    _, hl = ss.ss_scan_fwd(u, u, A, B, B, return_last_state=True, h0=h0)
    torch.cuda.synchronize()
    assert torch.equal(hl, h0)


# --- the row-sequential kernel: rows (Bsz * Dch) >= 8192 with L a multiple of
# the 16-byte vector select it; tiles are 32 steps, CTAs 32 channels.
ROWS_SHAPES = [
    (4, 2080, 200),  # channels not a multiple of the CTA, a ragged last tile
    (8, 1040, 32),   # exactly one tile
    (2, 4100, 8),    # less than one tile
    (1, 8200, 72),   # one batch, two full tiles and a part
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("Bsz,Dch,L", ROWS_SHAPES)
def test_rows_kernel_shapes(dtype, Bsz, Dch, L):
    x = make_case(dtype, Bsz, Dch, L, seed=300 + L + Dch)
    compare(x, dtype, what=f"rows {dtype} {Bsz}x{Dch}x{L}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("drop", ["D", "z", "delta_bias", "all", "softplus"])
def test_rows_kernel_optional_inputs(dtype, drop):
    x = make_case(dtype, 4, 2060, 96, seed=17)
    softplus = True
    if drop == "all":
        x.update(D=None, z=None, delta_bias=None)
    elif drop == "softplus":
        softplus = False
        x["delta"] = as_io(np.abs(synth.widen(x["delta"])) * 0.05, dtype)
        x["delta_bias"] = np.zeros_like(x["delta_bias"])
    else:
        x[drop] = None
    compare(x, dtype, softplus=softplus, what=f"rows {dtype} drop={drop}")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_rows_kernel_from_state_in_place(dtype):
    """Row-sequential kernel continued from a state updated in place."""
    Bsz, Dch, L = 4, 2070, 136
    x = make_case(dtype, Bsz, Dch, L, seed=71)
    h0 = np.random.default_rng(9).standard_normal((Bsz, Dch, 16)).astype(np.float32)
    xd = inputs_to_dev(x, dtype)
    h = torch.from_numpy(h0).cuda()
    y, hl = ss.ss_scan_fwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                           xd["delta_bias"], True, return_last_state=True, h0=h, h_last=h)
    torch.cuda.synchronize()
    assert hl.data_ptr() == h.data_ptr()
    ref, href = oracle_fwd(x, True, h0=h0.astype(np.float64))
    check(to_host64(y), ref, out_kind(dtype), f"rows {dtype} from state y")
    check(to_host64(hl), href, "f32", "rows h_last")


def test_rows_kernel_deterministic():
    x = make_case("bf16", 4, 2048, 160, seed=12)
    xd = inputs_to_dev(x, "bf16")
    y1, h1 = run_fwd(xd)
    y2, h2 = run_fwd(xd)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(h1, h2)
