"""Host-side pieces of bench.py (no GPU): the method's work counts per
scanned element and the roofline arithmetic that the JSON line reports."""
import math

import bench


def test_forward_work_counts():
    w = bench.method_work("fwd", 2, 1536)
    # per element: u, delta, z in and y out (bf16) plus B, C once per (b, t)
    assert math.isclose(w["bytes"], 8 + 2 * 16 * 2 / 1536)
    assert w["mufu"] == 16 + 4 and w["fp32"] == 4 * 16 + 10


def test_backward_is_the_method_total_less_the_forward():
    N = 16
    f, b, fb = (bench.method_work(k, 4, 2048, N) for k in ("fwd", "bwd", "fwd_bwd"))
    assert b["fp32"] == (14 * N + 20) - (4 * N + 10) == 10 * N + 10
    assert b["mufu"] == N + 6
    assert fb["fp32"] == f["fp32"] + b["fp32"] and fb["mufu"] == f["mufu"] + b["mufu"]
    # fp32 I/O: u, delta, z, dy in, du, ddelta, dz out; B, C in, dB, dC out
    assert math.isclose(b["bytes"], 7 * 4 + (2 * N * 4 + 8 * N) / 2048)


def test_work_scales_with_state_size():
    w16, w64 = bench.method_work("fwd", 2, 1536, 16), bench.method_work("fwd", 2, 1536, 64)
    assert w64["mufu"] - w16["mufu"] == 48 and w64["fp32"] - w16["fp32"] == 4 * 48


def test_step_work_is_per_token_row():
    w = bench.method_work("step", 2, 5120)
    # the float32 state read and written, u, delta, z in and y out, B and C
    assert math.isclose(w["bytes"], 8 * 16 + 8 + 2 * 16 * 2 / 5120)


def test_peaks_from_per_sm_rates():
    p = bench.Peaks({"ffma": 128.0, "ex2": 32.0})
    assert math.isclose(p.fp32_t, 148 * 128 * 2032e6 / 1e12)
    assert math.isclose(p.mufu_t, 148 * 32 * 2032e6 / 1e12)
    assert p.pipes_src == "measured"
    assert bench.Peaks(None).pipes_src == "fallback"


def test_roofline_picks_the_slowest_resource():
    E = 8 * 1536 * 2048
    p = bench.Peaks({"ffma": 128.0, "ex2": 32.0})
    r = bench.roofline(dict(fp32=0, mufu=0, bytes=4.0), E, 0.1, p)  # memory only
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert math.isclose(r["achieved"], round(4.0 * E / 1e-4 / 1e9, 1))
    assert math.isclose(r["frac"], round(r["achieved"] / p.hbm_gbs, 4), abs_tol=1e-4)
    r = bench.roofline(dict(fp32=1000, mufu=1, bytes=1.0), E, 1.0, p)  # FP32 dominates
    assert r["bound"] == "alu" and r["resource"] == "fp32" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["peak"], round(p.fp32_t, 3))
    r = bench.roofline(dict(fp32=1, mufu=100, bytes=1.0), E, 1.0, p)  # MUFU dominates
    assert r["resource"] == "mufu"
    assert math.isclose(r["frac"], round(100 * E / 1e-3 / 1e12 / p.mufu_t, 4))


def test_kernel_digest_ignores_comments_only():
    """The ncu figures stay attached to a kernel while its code is unchanged:
    comments and blank lines do not count, code does."""
    src = "// header\nint f(int x) {  // trailing\n  /* block\n  comment */ return x + 1;\n}\n"
    same = "int f(int x) {\n\n  return x + 1;   \n}\n// new note\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
