"""Host-side pieces of bench.py (no GPU): the algorithmic work counts and the
roofline arithmetic that the JSON line reports."""
import math

import bench


def test_forward_work_counts():
    w = bench.kernel_work(2, 1536)["fwd"]
    # per element: u, delta, z in and y out (bf16) plus B, C once per (b, t)
    assert math.isclose(w["bytes"], 8 + 2 * 16 * 2 / 1536)
    assert w["mufu"] == 16 + 4 and w["fp32"] == 4 * 16 + 9


def test_work_scales_with_state_size():
    w16, w64 = bench.kernel_work(2, 1536, 16), bench.kernel_work(2, 1536, 64)
    assert w64["fwd"]["mufu"] - w16["fwd"]["mufu"] == 48
    assert w64["bwd_reverse"]["fp32"] - w16["bwd_reverse"]["fp32"] == 12 * 48


def test_roofline_picks_the_slowest_resource():
    E = 8 * 1536 * 2048
    work = dict(fp32=0, mufu=0, bytes=4.0)           # memory only
    r = bench.roofline("x", work, E, 0.1, 6500.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert math.isclose(r["achieved"], round(4.0 * E / 1e-4 / 1e9, 1))
    assert math.isclose(r["frac"], round(r["achieved"] / 6500.0, 4), abs_tol=1e-4)
    work = dict(fp32=1000, mufu=1, bytes=1.0)        # FP32 dominates
    r = bench.roofline("x", work, E, 1.0, 6500.0)
    assert r["bound"] == "alu" and r["resource"] == "fp32" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["peak"], round(bench.FP32_PEAK_T, 3))


def test_peaks_are_the_stated_unit_counts():
    assert math.isclose(bench.FP32_PEAK_T, 148 * 128 * 2032e6 / 1e12)
    assert math.isclose(bench.MUFU_PEAK_T, 148 * 32 * 2032e6 / 1e12)
