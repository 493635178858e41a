"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments with the documented status codes
before touching CUDA (so these calls are safe on a machine without a GPU)."""
import ctypes
import os
import re

import pytest

import selective_state_space_114_b300 as ss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "selscan.h")

OK, NULL, SHAPE, DTYPE, NUNS, ALIGN, WS = 0, 1, 2, 3, 4, 5, 6


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    assert declared_functions() == sorted(ss.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(ss.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for code in range(10):
        s = ss.ss_status_str(code)
        assert s and s.startswith("SS_")
    assert ss.ss_status_str(ss.SS_ERR_TIMEOUT).startswith("SS_ERR_TIMEOUT")
    assert ss.ss_status_str(99) == "unknown ss_status"
    assert ss.ss_version() >= 10000


# Fake "device" addresses: never dereferenced, the calls below are rejected first.
P = 0x10000
MIS = 0x10004


def fwd(**kw):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, softplus=1, Bsz=2, Dch=16,
             L=64, N=16, dtype=0, y=P, h_last=None)
    a.update(kw)
    return ss.lib().ss_scan_fwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["bias"], a["softplus"], a["Bsz"], a["Dch"], a["L"], a["N"],
                                a["dtype"], a["y"], a["h_last"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), DTYPE),
    (dict(N=12), NUNS),
    (dict(N=128), NUNS),
    (dict(L=-1), SHAPE),
    (dict(Bsz=-3), SHAPE),
    (dict(Bsz=70000), SHAPE),
    (dict(Dch=1 << 41), SHAPE),
    (dict(u=None), NULL),
    (dict(B=None), NULL),
    (dict(y=None), NULL),
    (dict(A=None), NULL),
    (dict(u=MIS), ALIGN),
    (dict(D=MIS), ALIGN),
    (dict(h_last=MIS), ALIGN),
])
def test_fwd_rejects(kw, code):
    assert fwd(**kw) == code


def test_fwd_empty_is_ok_without_pointers():
    assert fwd(u=None, delta=None, A=None, B=None, C=None, y=None, L=0) == OK
    assert fwd(u=None, delta=None, A=None, B=None, C=None, y=None, Bsz=0) == OK


def test_workspace_size():
    n = ctypes.c_size_t(0)
    f = ss.lib().ss_scan_bwd_workspace_size
    assert f(8, 2048, 2048, 16, 0, ctypes.byref(n)) == OK and n.value > 0
    big = n.value
    assert f(8, 2048, 4096, 16, 0, ctypes.byref(n)) == OK and n.value > big
    assert f(0, 2048, 2048, 16, 0, ctypes.byref(n)) == OK and n.value == 0
    assert f(8, 2048, 2048, 12, 0, ctypes.byref(n)) == NUNS
    assert f(8, 2048, 2048, 64, 0, ctypes.byref(n)) == OK and n.value > big
    assert f(8, 2048, 2048, 16, 9, ctypes.byref(n)) == DTYPE
    assert f(8, 2048, 2048, 16, 0, None) == NULL
    assert ss.ss_scan_bwd_workspace_size(2, 16, 64) % 256 == 0


def bwd(**kw):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=P, z=P, bias=P, softplus=1, dy=P, Bsz=2, Dch=16,
             L=64, N=16, dtype=1, du=P, dd=P, dA=P, dB=P, dC=P, dD=P, dz=P, dbias=P, ws=P,
             wsb=1 << 30)
    a.update(kw)
    return ss.lib().ss_scan_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["bias"], a["softplus"], a["dy"], a["Bsz"], a["Dch"], a["L"],
                                a["N"], a["dtype"], a["du"], a["dd"], a["dA"], a["dB"], a["dC"],
                                a["dD"], a["dz"], a["dbias"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), DTYPE),
    (dict(N=4), NUNS),
    (dict(N=48), NUNS),
    (dict(L=-5), SHAPE),
    (dict(dy=None), NULL),
    (dict(dB=None), NULL),
    (dict(dD=None), NULL),          # D given but no dD
    (dict(z=None), NULL),           # dz given but no z
    (dict(bias=None), NULL),        # ddelta_bias given but no delta_bias
    (dict(du=MIS), ALIGN),
    (dict(ws=None), WS),
    (dict(ws=MIS), WS),
    (dict(wsb=1000), WS),
])
def test_bwd_rejects(kw, code):
    assert bwd(**kw) == code


def step(**kw):
    a = dict(h=P, u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, softplus=1, Bsz=4,
             Dch=8, N=16, dtype=1, y=P)
    a.update(kw)
    return ss.lib().ss_step(a["h"], a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                            a["bias"], a["softplus"], a["Bsz"], a["Dch"], a["N"], a["dtype"],
                            a["y"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=3), DTYPE),
    (dict(N=128), NUNS),
    (dict(N=4), NUNS),
    (dict(Dch=-1), SHAPE),
    (dict(Bsz=65536), SHAPE),
    (dict(h=None), NULL),
    (dict(y=None), NULL),
    (dict(h=MIS), ALIGN),
    (dict(B=MIS), ALIGN),
])
def test_step_rejects(kw, code):
    assert step(**kw) == code


def test_step_empty_is_ok():
    assert step(h=None, u=None, delta=None, A=None, B=None, C=None, y=None, Bsz=0) == OK


def fwd_from_state(**kw):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, softplus=1, h0=P, Bsz=2,
             Dch=16, L=64, N=16, dtype=0, y=P, h_last=None)
    a.update(kw)
    return ss.lib().ss_scan_fwd_from_state(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"],
                                           a["z"], a["bias"], a["softplus"], a["h0"], a["Bsz"],
                                           a["Dch"], a["L"], a["N"], a["dtype"], a["y"],
                                           a["h_last"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), DTYPE), (dict(N=24), NUNS), (dict(L=-1), SHAPE), (dict(u=None), NULL),
    (dict(h0=MIS), ALIGN),
])
def test_fwd_from_state_rejects(kw, code):
    assert fwd_from_state(**kw) == code


def conv(**kw):
    a = dict(x=P, w=P, bias=None, silu=1, Bsz=2, Dch=16, L=64, K=4, dtype=1, u=P)
    a.update(kw)
    return ss.lib().ss_conv1d_silu_fwd(a["x"], a["w"], a["bias"], a["silu"], a["Bsz"], a["Dch"],
                                       a["L"], a["K"], a["dtype"], a["u"], None)


def conv_bwd(**kw):
    a = dict(x=P, w=P, bias=P, silu=1, du=P, Bsz=2, Dch=16, L=64, K=4, dtype=1, dx=P, dw=P,
             dbias=P)
    a.update(kw)
    return ss.lib().ss_conv1d_silu_bwd(a["x"], a["w"], a["bias"], a["silu"], a["du"], a["Bsz"],
                                       a["Dch"], a["L"], a["K"], a["dtype"], a["dx"], a["dw"],
                                       a["dbias"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), SHAPE), (dict(K=5), SHAPE), (dict(L=-2), SHAPE), (dict(dtype=9), DTYPE),
    (dict(x=None), NULL), (dict(w=None), NULL), (dict(u=None), NULL), (dict(x=MIS), ALIGN),
    (dict(u=MIS), ALIGN),
])
def test_conv_rejects(kw, code):
    assert conv(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(K=7), SHAPE), (dict(dtype=4), DTYPE), (dict(du=None), NULL), (dict(dw=None), NULL),
    (dict(dbias=None), NULL), (dict(bias=None), NULL), (dict(dx=MIS), ALIGN),
])
def test_conv_bwd_rejects(kw, code):
    assert conv_bwd(**kw) == code


def test_conv_empty_forward_is_ok_without_pointers():
    assert conv(x=None, w=None, u=None, L=0) == OK


def xproj(**kw):
    a = dict(u=P, Wx=P, Wdt=P, Bsz=2, Dch=64, L=128, R=16, N=8, dtype=1, delta=P, B=P, C=P)
    a.update(kw)
    return ss.lib().ss_xproj(a["u"], a["Wx"], a["Wdt"], a["Bsz"], a["Dch"], a["L"], a["R"], a["N"],
                             a["dtype"], a["delta"], a["B"], a["C"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=0), DTYPE), (dict(dtype=7), DTYPE), (dict(R=4), SHAPE), (dict(R=12), SHAPE),
    (dict(N=0), SHAPE), (dict(R=160, N=56), SHAPE), (dict(L=100), SHAPE), (dict(Dch=60), SHAPE),
    (dict(L=-8), SHAPE), (dict(u=None), NULL), (dict(C=None), NULL), (dict(Wx=MIS), ALIGN),
    (dict(delta=MIS), ALIGN),
])
def test_xproj_rejects(kw, code):
    assert xproj(**kw) == code


def test_xproj_empty_is_ok_without_pointers():
    assert xproj(u=None, Wx=None, Wdt=None, delta=None, B=None, C=None, L=0) == OK


def noalloc(**kw):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=P, z=P, bias=P, softplus=1, dy=P, Bsz=2, Dch=16,
             L=64, N=16, dtype=1, du=P, dd=P, dA=P, dB=P, dC=P, dD=P, dz=P, dbias=P)
    a.update(kw)
    return ss.lib().ss_scan_bwd_noalloc(
        a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"], a["softplus"],
        a["dy"], a["Bsz"], a["Dch"], a["L"], a["N"], a["dtype"], a["du"], a["dd"], a["dA"],
        a["dB"], a["dC"], a["dD"], a["dz"], a["dbias"], None)


BIG = dict(Bsz=4, Dch=1024, L=4096)  # needs more than the 32 MiB static buffer


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), DTYPE),
    (dict(N=4), NUNS),
    (dict(dy=None), NULL),
    (dict(dD=None), NULL),
    (dict(du=MIS), ALIGN),
    # ss_scan_bwd's argument checks come before the scratch limit
    (dict(dy=None, **BIG), NULL),
    (dict(du=MIS, **BIG), ALIGN),
    (dict(BIG), 8),                 # SS_ERR_SCRATCH_LIMIT
])
def test_noalloc_rejects_like_ss_scan_bwd_then_by_size(kw, code):
    assert noalloc(**kw) == code


def test_check_device_errors_without_a_device_reports_a_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("covered by the GPU tests")
    assert ss.lib().ss_check_device_errors(None) == 7  # SS_ERR_CUDA
