"""Plants plausible mistakes in copies of the oracle source (on the CPU) and
checks that the pin suite rejects every one of them."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (original fragment, mutated fragment)
MUTATIONS = {
    "readout_before_update": ("          h[n] = dA * h[n] + dBu;\n          s += Ct[n] * h[n];",
                              "          s += Ct[n] * h[n];\n          h[n] = dA * h[n] + dBu;"),
    "A_transposed": ("exp(dt * A[d * d_state + n]);\n          double dBu = dt * Bt[n]",
                     "exp(dt * A[n * d_inner + d]);\n          double dBu = dt * Bt[n]"),
    "drop_skip_term": ("        if (D) s += D[d] * u[e];", ""),
    "no_delta_in_input_term": ("double dBu = dt * Bt[n] * u[e];", "double dBu = Bt[n] * u[e];"),
    "euler_discretisation": ("double dA = exp(dt * A[d * d_state + n]);\n          double dBu = dt * Bt[n]",
                             "double dA = 1.0 + dt * A[d * d_state + n];\n          double dBu = dt * Bt[n]"),
    "sigmoid_instead_of_silu": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "bias_after_softplus": (
        "  double x = delta_raw + (delta_bias ? delta_bias[d] : 0.0);\n  return softplus_flag ? oracle_softplus(x) : x;",
        "  double x = softplus_flag ? oracle_softplus(delta_raw) : delta_raw;\n  return x + (delta_bias ? delta_bias[d] : 0.0);"),
    "readout_with_B": ("s += Ct[n] * h[n];\n        }\n        if (D) s += D[d] * u[e];",
                       "s += Bt[n] * h[n];\n        }\n        if (D) s += D[d] * u[e];"),
    "softplus_sign": ("if (x > 0.0) return x + log1p(exp(-x));", "if (x > 0.0) return x - log1p(exp(-x));"),
    "last_state_index": ("last_state[(b * d_inner + d) * d_state + n] = h[n];",
                         "last_state[(d * batch + b) * d_state + n] = h[n];"),
    "gate_dropped": ("        if (z) s *= oracle_silu(z[e]);\n        y[e] = s;", "        y[e] = s;"),
    "initial_state_ignored": ("        h[n] = initial_state ? initial_state[(b * d_inner + d) * d_state + n] : 0.0;",
                              "        h[n] = 0.0;"),
    "conv_taps_reversed": ("          acc += w[d * d_conv + k] * xv;",
                           "          acc += w[d * d_conv + (d_conv - 1 - k)] * xv;"),
    "conv_history_shifted": ("else if (x_prev) xv = x_prev[(b * d_inner + d) * (d_conv - 1) + (s + d_conv - 1)];",
                             "else if (x_prev) xv = x_prev[(b * d_inner + d) * (d_conv - 1) + (s + d_conv - 2)];"),
    "bwd_carry_without_decay": ("          lam[n] *= dAn;                         /* carry dA_t lambda_t to step t-1 */",
                                "          lam[n] *= 1.0;"),
    "bwd_dB_without_step": ("dB[(b * L + t) * N + n] += lam[n] * dt * u[e];",
                            "dB[(b * L + t) * N + n] += lam[n] * u[e];"),
    "bwd_dC_previous_state": ("dC[(b * L + t) * N + n] += ds * h[n];", "dC[(b * L + t) * N + n] += ds * hp[n];"),
    "bwd_softplus_derivative": ("const double dx = softplus_flag ? ddt * oracle_sigmoid(x) : ddt;",
                                "const double dx = softplus_flag ? ddt * oracle_sigmoid(-x) : ddt;"),
    "decode_no_decay": ("      double dA = exp(dt * A[d * d_state + n]);\n      double dBu = dt * Bb[n] * u[ch];",
                        "      double dA = 1.0;\n      double dBu = dt * Bb[n] * u[ch];"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutation(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "ssm_oracle.c")).read()
    before, after = MUTATIONS[name]
    assert before in src, f"mutation anchor for {name} not found"
    work = tmp_path / "repo"
    shutil.copytree(os.path.join(ROOT, "oracle"), work / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests"), work / "tests",
                    ignore=shutil.ignore_patterns("__pycache__"))
    (work / "oracle" / "ssm_oracle.c").write_text(src.replace(before, after, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=work, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
