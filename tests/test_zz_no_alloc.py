"""ss_scan_bwd_noalloc: the backward scan for callers that cannot allocate.

Some callers cannot call cudaMalloc (a plugin inside an application that
owns all device memory, or a loop that must never enter the allocator).
This entry point takes no workspace; it uses a static scratch buffer inside
the library instead.  It runs the same kernels as ss_scan_bwd, so its results
must equal ss_scan_bwd's bit for bit, on consecutive calls that leave
different contents in the shared buffer; the first call is also checked
against the fp64 oracle.  Problems larger than the buffer must be refused
before anything runs.

Called through the C ABI (ctypes), not through a Python wrapper.
"""
import ctypes

import pytest
import torch

from parity_util import check, grad_kind, inputs_to_dev, make_case, oracle_bwd, to_dev, to_host64

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

SS_OK, SS_ERR_SCRATCH_LIMIT = 0, 8
IO = ("du", "ddelta", "dz")
NAMES = ("du", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddelta_bias")


def _alloc_grads(xd):
    u = xd["u"]
    Bsz, Dch, L = u.shape
    dev = u.device
    return {"du": torch.empty_like(u), "ddelta": torch.empty_like(u), "dz": torch.empty_like(u),
            "dA": torch.empty((Dch, 16), device=dev), "dB": torch.empty((Bsz, 16, L), device=dev),
            "dC": torch.empty((Bsz, 16, L), device=dev), "dD": torch.empty((Dch,), device=dev),
            "ddelta_bias": torch.empty((Dch,), device=dev)}


def _noalloc(xd, dyd, g):
    u = xd["u"]
    Bsz, Dch, L = u.shape
    code = ss.SS_BF16 if u.dtype == torch.bfloat16 else ss.SS_F32
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return ss.lib().ss_scan_bwd_noalloc(
        p(u), p(xd["delta"]), p(xd["A"]), p(xd["B"]), p(xd["C"]), p(xd["D"]), p(xd["z"]),
        p(xd["delta_bias"]), 1, p(dyd), Bsz, Dch, L, 16, code, p(g["du"]), p(g["ddelta"]),
        p(g["dA"]), p(g["dB"]), p(g["dC"]), p(g["dD"]), p(g["dz"]), p(g["ddelta_bias"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(dtype, Bsz, Dch, L, seed, host=False):
    x = make_case(dtype, Bsz, Dch, L, seed=seed, with_dy=True)
    dy = x.pop("dy")
    dev = (inputs_to_dev(x, dtype), to_dev(dy, dtype))
    return dev + (x, dy) if host else dev


def test_noalloc_matches_workspace_backward_on_consecutive_calls():
    limit = ss.lib().ss_scan_bwd_noalloc_max_scratch()
    assert limit == 32 << 20
    # the second call runs on a smaller problem, over the first call's leftovers
    cases = [("bf16", 3, 40, 1000, 41), ("f32", 2, 17, 300, 43)]
    for i, (dtype, Bsz, Dch, L, seed) in enumerate(cases):
        assert ss.ss_scan_bwd_workspace_size(Bsz, Dch, L) <= limit
        xd, dyd, x, dy = _case(dtype, Bsz, Dch, L, seed, host=True)
        g = _alloc_grads(xd)
        assert _noalloc(xd, dyd, g) == SS_OK
        ref = ss.ss_scan_bwd(xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd["D"], xd["z"],
                             xd["delta_bias"], True, dyd)
        torch.cuda.synchronize()
        for k in NAMES:
            assert torch.equal(g[k], ref[k]), f"noalloc {dtype} {k} differs from ss_scan_bwd"
        if i == 0:  # and against the fp64 oracle on the same inputs
            oref = oracle_bwd(x, dy, True)
            for k in NAMES:
                check(to_host64(g[k]), oref[k], grad_kind(dtype, k in IO), f"noalloc {dtype} {k}")


def test_noalloc_refuses_problems_larger_than_its_buffer():
    limit = ss.lib().ss_scan_bwd_noalloc_max_scratch()
    Bsz, Dch, L = 4, 1024, 4096
    assert ss.ss_scan_bwd_workspace_size(Bsz, Dch, L) > limit
    xd, dyd = _case("bf16", Bsz, Dch, L, 47)
    g = {k: v.fill_(3.0) for k, v in _alloc_grads(xd).items()}
    assert _noalloc(xd, dyd, g) == SS_ERR_SCRATCH_LIMIT
    assert "SCRATCH" in ss.ss_status_str(SS_ERR_SCRATCH_LIMIT)
    torch.cuda.synchronize()
    for k, v in g.items():
        assert torch.all(v == 3.0), k
