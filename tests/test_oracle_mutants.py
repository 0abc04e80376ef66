"""Plant plausible mistakes in a copy of the oracle source (CPU only) and check that the
pins catch every one of them.  The built oracle itself is never modified."""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, exact text in the oracle source, replacement)
MUTANTS = [
    ("no_decay", "S[(size_t)d * V + j] *= decay;", "(void)decay;"),
    ("delta_sign", "(vt[j] - r[j])", "(r[j] - vt[j])"),
    ("no_beta", "bt * kt[d] * (vt[j] - r[j])", "kt[d] * (vt[j] - r[j])"),
    ("readout_transposed", "acc += S[(size_t)d * V + j] * (qt[d] * qs);",
     "acc += S[(size_t)j * V + d] * (qt[d] * qs);"),
    ("nonsafe_sign", "return -exp(A_log) * softplus(g + dt_bias);",
     "return exp(A_log) * softplus(g + dt_bias);"),
    ("nonsafe_no_exp_A", "return -exp(A_log) * softplus(g + dt_bias);",
     "return -A_log * softplus(g + dt_bias);"),
    ("softplus_relu", "return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));",
     "return x > 0.0 ? x : log1p(exp(x));"),
    ("knorm_no_sqrt", "const double ks = 1.0 / sqrt(ss + k_eps);", "const double ks = 1.0 / (ss + k_eps);"),
    ("beta_logit_sign", "1.0 / (1.0 + exp(-braw))", "1.0 / (1.0 + exp(braw))"),
    ("gva_heads_interleaved", "const int hk = h / (H / Hk);", "const int hk = h % Hk;"),
    ("qnorm_no_sqrt", "qs = 1.0 / sqrt(ss + q_eps);", "qs = 1.0 / (ss + q_eps);"),
    ("qnorm_no_eps", "qs = 1.0 / sqrt(ss + q_eps);", "qs = 1.0 / sqrt(ss);"),
    ("qnorm_abs_sum", "ss += qt[d] * qt[d];", "ss += fabs(qt[d]);"),
    ("no_scale", "ot[j] = acc * scale;", "ot[j] = acc;"),
    ("r_uses_q", "r[j] += S[(size_t)d * V + j] * kt[d];", "r[j] += S[(size_t)d * V + j] * qt[d];"),
    ("sigmoid_sign", "exp(-z)", "exp(z)"),
    ("no_dt_bias", "double z = exp(A_log) * (g + dt_bias);", "double z = exp(A_log) * g;"),
    ("no_exp_A", "double z = exp(A_log) * (g + dt_bias);", "double z = A_log * (g + dt_bias);"),
    ("log2_gate_unscaled", "return g * ORC_LN2;", "return g;"),
    ("no_initial_state", "if (S0) memcpy(S, S0 + st_off", "if (0) memcpy(S, S0 + st_off"),
    ("no_chunk_reset", "if ((t - bos) % chunk_size == 0) acc = 0.0;", ";"),
    ("gate_natural_units", "out[idx] = acc / ORC_LN2;", "out[idx] = acc;"),
    ("decay_wrong_channel", "double decay = exp(kda_oracle_gate_act(gt[d],",
     "double decay = exp(kda_oracle_gate_act(gt[0],"),
    ("varlen_short_by_one", "*eos = cu[n + 1]; }", "*eos = cu[n + 1] - (cu[n + 1] > cu[n]); }"),
    ("dense_rows_shifted", "*bos = (long)n * T; *eos = (long)n * T + T;",
     "*bos = (long)n * T; *eos = (long)n * T + T - 1;"),
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_dir, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = os.path.join(mutant_dir, f"{name}.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    so = os.path.join(mutant_dir, f"lib_{name}.so")
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", so, src, "-lm"],
                   check=True, capture_output=True)
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib=lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
