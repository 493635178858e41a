"""The seeded input generator (CPU only): determinism, element-wise
regeneration, distributions and bf16 rounding."""
import numpy as np

import synth


def test_deterministic_and_indexable():
    a = synth.normal(1000, 1, 50_000, "f32")
    b = synth.normal(1000, 1, 50_000, "f32")
    assert np.array_equal(a, b)
    idx = np.array([0, 17, 49_999])
    assert np.array_equal(synth.normal_at(1000, 1, idx), a[idx])
    assert np.array_equal(synth.normal(1000, 1, 100, "f32", start=300), a[300:400])
    assert not np.array_equal(a, synth.normal(1001, 1, 50_000, "f32"))
    assert not np.array_equal(a, synth.normal(1000, 2, 50_000, "f32"))


def test_normal_moments():
    x = synth.normal(7, 3, 400_000, "f32").astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    assert abs(np.mean(x ** 3)) < 0.02 and abs(np.mean(x ** 4) - 3) < 0.05


def test_bf16_round_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    bits = synth.to_bf16(f)
    got = synth.widen(bits)
    # ties go to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> 1.0
    assert list(got) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]
    x = synth.normal(5, 1, 10_000, "f32")
    xb = synth.widen(synth.normal(5, 1, 10_000, "bf16"))
    assert np.all(np.abs(xb - x) <= np.abs(x) * 2 ** -8 + 1e-30)


def test_delta_bias_is_inverse_softplus_of_log_uniform_dt():
    lo, hi = 1e-3, 1e-1
    bias = synth.param_delta_bias(1000, 4096, (lo, hi)).astype(np.float64)
    dt = np.logaddexp(0.0, bias)
    assert dt.min() >= lo * 0.999 and dt.max() <= hi * 1.001
    # log-uniform: log dt is uniform over [log lo, log hi]
    q = (np.log(dt) - np.log(lo)) / (np.log(hi) - np.log(lo))
    assert abs(q.mean() - 0.5) < 0.02


def test_row_inputs_match_full_tensors():
    cfg = synth.config(0)
    full = synth.make_inputs(cfg)
    r = synth.row_inputs(cfg, 1, 5)
    for k in ("u", "delta", "z"):
        assert np.array_equal(r[k], full[k][1, 5])
    for k in ("B", "C"):
        assert np.array_equal(r[k], full[k][1])
    assert np.array_equal(r["A"], full["A"][5])
    assert np.array_equal(r["delta_bias"], full["delta_bias"][5:6])
