"""The timeout path of a bounded device wait, without faulting or hanging.

ss_xproj waits on tensor-core completion barriers, each wait bounded.  The
test hook ss_debug_xproj_stuck_wait makes every CTA also wait (64 polls) on a
barrier nothing ever completes, so that wait gives up: the CTA sets the
device error word, waits for the tensor-core work it already issued, frees
its tensor memory and returns.  ss_check_device_errors must then report
SS_ERR_TIMEOUT once, and the next ordinary call must run correctly on the same
context."""
import pytest
import torch

import selective_state_space_114_b300 as ss
from test_parity_xproj import check_xproj, make

pytestmark = pytest.mark.gpu


def _run(u, Wx, Wdt, N):
    bf = lambda a: torch.from_numpy(a.copy()).view(torch.bfloat16).cuda()
    out = ss.ss_xproj(bf(u), bf(Wx), bf(Wdt), N)
    torch.cuda.synchronize()
    return out


def test_stuck_wait_reports_timeout_and_the_context_stays_usable():
    u, Wx, Wdt = make("bf16", 2, 200, 136, 48, 16, seed=71)
    assert ss.ss_check_device_errors() == ss.SS_OK  # clear anything earlier
    before = ss.ss_xproj_wait_failures()
    ss.ss_debug_xproj_stuck_wait(True)
    try:
        _run(u, Wx, Wdt, 16)
    finally:
        ss.ss_debug_xproj_stuck_wait(False)
    assert ss.ss_check_device_errors() == ss.SS_ERR_TIMEOUT
    assert ss.ss_check_device_errors() == ss.SS_OK  # the check clears the word
    assert ss.ss_xproj_wait_failures() > before
    # the same context runs the next call normally
    got = _run(u, Wx, Wdt, 16)
    check_xproj(u, Wx, Wdt, 16, "bf16", got, "after a timeout")
    assert ss.ss_check_device_errors() == ss.SS_OK
