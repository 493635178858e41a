"""Each pin must be able to fail: plant a plausible mistake in a copy of the
oracle's C source (on the CPU, never in the CUDA path), build it, and check
that at least one pin rejects the mutant."""
import os

import pytest

import oracle
import oracle_pins

# (name, original text, mutated text); each original must occur in oracle.c
MUTANTS = [
    ("euler_A_instead_of_zoh", "const double dA = exp(dt * A[n]);", "const double dA = 1.0 + dt * A[n];"),
    ("dBu_scaled_by_dA", "h[n] = dA * h[n] + dBu;", "h[n] = dA * h[n] + dBu * dA;"),
    ("C_swapped_for_B", "y += Cb[n * L + t] * h[n];", "y += Bb[n * L + t] * h[n];"),
    ("skip_uses_delta", "y += Dd * u[t];", "y += Dd * dr[t];"),
    ("softplus_unstable_branch", "return fmax(x, 0.0) + log1p(exp(-fabs(x)));",
     "return fmax(x, 0.0) + log1p(exp(-x));"),
    ("gate_sigmoid_only", "if (z) y = y * z[t] * sigmoid(z[t]);", "if (z) y = y * sigmoid(z[t]);"),
    ("bias_dropped", "const double dt = softplus_or_raw(dr[t] + bias, c->softplus);",
     "const double dt = softplus_or_raw(dr[t], c->softplus);"),
    ("B_row_by_channel", "const double* Bb = c->B + b * N * L;\n    const double* Cb = c->C + b * N * L;\n    const double* A = c->A + d * N;\n    const double Dd = c->D ? c->D[d] : 0.0;\n    const double bias = c->bias ? c->bias[d] : 0.0;\n    double h[1024];",
     "const double* Bb = c->B + (d % c->Bsz) * N * L;\n    const double* Cb = c->C + b * N * L;\n    const double* A = c->A + d * N;\n    const double Dd = c->D ? c->D[d] : 0.0;\n    const double bias = c->bias ? c->bias[d] : 0.0;\n    double h[1024];"),
    ("blelloch_operand_order", "eb[k] = la * pb + lb;", "eb[k] = pa * lb + pb;"),
    ("adjoint_uses_own_decay", "lam[n] = yhat[t] * Cb[n * L + t] + a_next * lam[n];",
     "lam[n] = yhat[t] * Cb[n * L + t] + Aa[t * N + n] * lam[n];"),
    ("ddelta_uses_h_t", "ddt += lam[n] * (h_prev * a_t * A[n] + Bt * u[t]);",
     "ddt += lam[n] * (h_t * a_t * A[n] + Bt * u[t]);"),
    ("ddelta_sign", "ddt += lam[n] * (h_prev * a_t * A[n] + Bt * u[t]);",
     "ddt += lam[n] * (h_prev * a_t * A[n] - Bt * u[t]);"),
    ("dA_drops_decay", "dA_acc[n] += lam[n] * h_prev * a_t * dt;", "dA_acc[n] += lam[n] * h_prev * dt;"),
    ("dz_wrong_derivative", "c->dz[row * L + t] = g[t] * y * s * (1.0 + z[t] * (1.0 - s));",
     "c->dz[row * L + t] = g[t] * y * s * (1.0 + z[t] * s);"),
    ("dbias_sigmoid_of_delta", "const double ddraw = c->softplus ? ddt * sigmoid(xs[t]) : ddt;",
     "const double ddraw = c->softplus ? ddt * sigmoid(dts[t]) : ddt;"),
    ("dB_drops_delta", "tdB[(b * N + n) * L + t] += lam[n] * dt * u[t];", "tdB[(b * N + n) * L + t] += lam[n] * u[t];"),
    ("dC_uses_h_prev", "tdC[(b * N + n) * L + t] += yhat[t] * h_t;", "tdC[(b * N + n) * L + t] += yhat[t] * h_prev;"),
    ("du_drops_delta", "du_t += lam[n] * dt * Bt;", "du_t += lam[n] * Bt;"),
    ("dD_ungated", "dD_acc += yhat[t] * u[t];", "dD_acc += g[t] * u[t];"),
    ("step_B_for_C", "y += c->C[b * N + n] * *hn;", "y += c->B[b * N + n] * *hn;"),
    ("step_no_bias", "const double dt = softplus_or_raw(c->delta[row] + (c->bias ? c->bias[d] : 0.0), c->softplus);",
     "const double dt = softplus_or_raw(c->delta[row], c->softplus);"),
    ("conv_taps_not_flipped", "if (src >= 0) s += c->w[d * c->K + k] * xr[src];",
     "if (src >= 0) s += c->w[d * c->K + (c->K - 1 - k)] * xr[src];"),
    ("conv_bias_dropped", "double s = c->bias ? c->bias[d] : 0.0;", "double s = 0.0;"),
    ("conv_silu_derivative_wrong", "c->g[row * L + t] * s * (1.0 + v * (1.0 - s))",
     "c->g[row * L + t] * s"),
    ("conv_dx_wrong_tap", "if (t < L) acc += c->w[d * K + k] * gc[t];",
     "if (t < L) acc += c->w[d * K + (K - 1 - k)] * gc[t];"),
    ("conv_dw_wrong_shift", "if (src >= 0) c->dw[d * K + k] += gc[t] * xr[src];",
     "if (src >= 1) c->dw[d * K + k] += gc[t] * xr[src - 1];"),
    ("xproj_weight_transposed", "s += c->Wx[m * c->Dch + k] * ub[k * c->L + t];",
     "s += c->Wx[(k % M) * c->Dch + (m % c->Dch)] * ub[k * c->L + t];"),
    ("xproj_B_C_swapped", "c->B[(b * c->N + n) * c->L + t] = x[c->R + n];",
     "c->B[(b * c->N + n) * c->L + t] = x[c->R + c->N + n];"),
    ("xproj_dt_part_shifted", "for (i64 r = 0; r < c->R; ++r) s += c->Wdt[d * c->R + r] * x[r];",
     "for (i64 r = 0; r < c->R; ++r) s += c->Wdt[d * c->R + r] * x[r + 1];"),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, mut, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(orig) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(orig, mut, 1)
    cpath = os.path.join(tmp_path, "oracle_mut.c")
    open(cpath, "w").write(mutated)
    so = oracle.compile_c(cpath, os.path.join(tmp_path, "liboracle_mut.so"))
    orc = oracle.Oracle(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError, RuntimeError) as e:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
