"""Forward that keeps the chunk states for its backward (ss_scan_fwd_save,
ss_scan_bwd_saved): the backward's gradients against the fp64 oracle and
against the backward that recomputes the states, on shapes that take each
forward kernel (the row-sequential kernel writes the states itself; the
chunked kernels get them from the backward's state summaries)."""
import numpy as np
import pytest
import torch

from parity_util import check, grad_kind, inputs_to_dev, make_case, oracle_bwd, to_dev, to_host64

import selective_state_space_114_b300 as ss

pytestmark = pytest.mark.gpu

IO_GRADS = ("du", "ddelta", "dz")
F32_GRADS = ("dA", "dB", "dC", "dD", "ddelta_bias")
STAGES = ("ss_scan_bwd_states", "ss_scan_bwd_reverse", "ss_scan_bwd_reduce")


def _ws(xd, N):
    Bsz, Dch, L = xd["u"].shape
    code = {torch.float32: ss.SS_F32, torch.bfloat16: ss.SS_BF16, torch.float16: ss.SS_F16}
    n = ss.ss_scan_bwd_workspace_size(Bsz, Dch, L, N, code[xd["u"].dtype])
    return torch.empty(max(n, 1), device="cuda", dtype=torch.uint8)


def _args(xd):
    return (xd["u"], xd["delta"], xd["A"], xd["B"], xd["C"], xd.get("D"), xd.get("z"),
            xd.get("delta_bias"), True)


@pytest.mark.parametrize("dtype,Bsz,Dch,L,N", [
    ("bf16", 2, 4096, 264, 16),   # row-sequential forward (8192 rows), ragged last chunk
    ("f32", 2, 4096, 136, 16),    # row-sequential, two rows per lane
    ("f16", 1, 8192, 96, 16),     # one partial chunk
    ("bf16", 2, 40, 520, 16),     # chunked paired forward: states from the summaries
    ("f32", 1, 24, 300, 16),      # chunked paired forward (fp32)
    ("bf16", 2, 33, 301, 16),     # element-wise forward
    ("bf16", 2, 48, 384, 8),      # other state sizes: row-sequential at any row count
    ("f32", 1, 40, 200, 32),
    ("bf16", 1, 20, 136, 64),
    ("bf16", 1, 16, 4500, 16),    # 36 chunks: the adjoint carry walks three blocks
    ("f32", 1, 24, 2200, 16),     # chunked forward, 18 chunks: state and adjoint carries
])
def test_saved_backward_matches_oracle_and_recompute(dtype, Bsz, Dch, L, N):
    x = make_case(dtype, Bsz, Dch, L, seed=900 + L + N, with_dy=True, N=N)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, dtype)
    dyd = to_dev(dy, dtype)
    ws = _ws(xd, N)
    y_plain = ss.ss_scan_fwd(*_args(xd))
    y_saved = ss.ss_scan_fwd(*_args(xd), save_to=ws)
    g_saved = ss.ss_scan_bwd(*_args(xd), dyd, workspace=ws, saved=True)
    g_plain = ss.ss_scan_bwd(*_args(xd), dyd)
    torch.cuda.synchronize()
    assert torch.equal(y_plain, y_saved), "saving the states must not change y"
    ref = oracle_bwd(x, dy, True)
    for k in IO_GRADS + F32_GRADS:
        got = to_host64(g_saved[k])
        check(got, ref[k], grad_kind(dtype, k in IO_GRADS), f"saved {dtype} {Bsz}x{Dch}x{L} N{N} {k}")
        # same gradients as the recomputing backward, up to rounding
        check(got, to_host64(g_plain[k]), grad_kind(dtype, k in IO_GRADS),
              f"saved vs recomputed {k}")


def test_saved_stagewise_equals_whole_saved_backward():
    x = make_case("bf16", 2, 4096, 256, seed=931, with_dy=True)
    dy = x.pop("dy")
    xd = inputs_to_dev(x, "bf16")
    dyd = to_dev(dy, "bf16")
    ws = _ws(xd, 16)
    ss.ss_scan_fwd(*_args(xd), save_to=ws)
    g1 = ss.ss_scan_bwd(*_args(xd), dyd, workspace=ws, saved=True)
    ss.ss_scan_fwd(*_args(xd), save_to=ws)  # the first backward reused the workspace
    g2 = ss.ss_scan_bwd(*_args(xd), dyd, workspace=ws, saved=True, stages=STAGES)
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_save_checks_the_workspace():
    x = make_case("f32", 2, 16, 300, seed=933)
    xd = inputs_to_dev(x, "f32")
    small = torch.empty(256, device="cuda", dtype=torch.uint8)
    with pytest.raises(ss.SelscanError) as e:
        ss.ss_scan_fwd(*_args(xd), save_to=small)
    assert e.value.status == 6  # SS_ERR_WORKSPACE
