"""Oracle pins (CPU) and a mutation test: every pin runs on the real oracle and must
pass; each deliberately broken copy of the oracle's C source must fail at least one."""
import os
import shutil
import tempfile

import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(oracle.default())


# (name, exact text in ssm_oracle.c, replacement): plausible mistakes.
MUTANTS = [
    ("sign_of_A", "double a = exp(dt * (double)A_d[n]);", "double a = exp(-dt * (double)A_d[n]);"),
    ("drop_D", "(D ? (double)D[d] * ut : 0.0)", "0.0"),
    ("B_for_C", "double bu = dt * (double)B_b[n * seqlen + t] * ut;",
     "double bu = dt * (double)C_b[n * seqlen + t] * ut;"),
    ("no_bias", "double x = (double)dl_r[t] + (delta_bias ? (double)delta_bias[d] : 0.0);",
     "double x = (double)dl_r[t];"),
    ("y_before_update", "h[n] = a * h[n] + bu;\n                acc += (double)C_b[n * seqlen + t] * h[n];",
     "acc += (double)C_b[n * seqlen + t] * h[n];\n                h[n] = a * h[n] + bu;"),
    ("sigmoid_gate", "yv *= oracle_silu((double)z_r[t]);", "yv *= 1.0 / (1.0 + exp(-(double)z_r[t]));"),
    ("no_softplus", "return x > 20.0 ? x : log1p(exp(x));", "return x;"),
    ("softplus_threshold", "return x > 20.0 ? x : log1p(exp(x));", "return x > 2.0 ? x : log1p(exp(x));"),
    ("ignore_h0", "h[n] = h0 ? h0[ch * dstate + n] : 0.0;", "h[n] = 0.0;"),
    ("B_time_shift", "double bu = dt * (double)B_b[n * seqlen + t] * ut;",
     "double bu = dt * (double)B_b[n * seqlen + (t > 0 ? t - 1 : 0)] * ut;"),
    ("zoh_like_Bbar", "double bu = dt * (double)B_b[n * seqlen + t] * ut;",
     "double bu = (double)B_b[n * seqlen + t] * ut;"),
    ("decode_drop_dt", "s[n] = a * s[n] + dt * (double)B[b * dstate + n] * xt;",
     "s[n] = a * s[n] + (double)B[b * dstate + n] * xt;"),
    ("h_last_zero", "h_last[ch * dstate + n] = h[n];", "h_last[ch * dstate + n] = 0.0;"),
    ("A_transposed", "const float *A_d = A + d * dstate;", "const float *A_d = A + d;"),
    ("conv_flipped", "acc += (double)w[d * width + k] * xp[t + k];",
     "acc += (double)w[d * width + (width - 1 - k)] * xp[t + k];"),
    ("conv_no_bias", "double acc = bias ? (double)bias[d] : 0.0;\n            for (int64_t k = 0; k < width; k++)",
     "double acc = 0.0;\n            for (int64_t k = 0; k < width; k++)"),
    ("conv_state_ignored", "xp[j] = conv_state_in ? conv_state_in[ch * hw + j] : 0.0;", "xp[j] = 0.0;"),
    ("conv_state_out_shift", "conv_state_out[ch * hw + j] = xp[seqlen + j];",
     "conv_state_out[ch * hw + j] = xp[seqlen + j - (j > 0)];"),
    ("conv_no_silu", "out[ch * seqlen + t] = silu ? oracle_silu(acc) : acc;", "out[ch * seqlen + t] = acc;"),
    ("conv_update_no_shift", "for (int64_t k = 0; k + 1 < hw; k++) s[k] = s[k + 1];", ""),
    ("bwd_no_softplus_grad", "if (softplus) dx = x > 20.0 ? ddt : ddt / (1.0 + exp(-x));", ""),
    ("bwd_no_decay_propagation", "g[n] *= an;", ""),
    ("bwd_dC_uses_prev_state", "dC_b[n * L + t] += dy * hs[(t + 1) * N + n];",
     "dC_b[n * L + t] += dy * hs[t * N + n];"),
    ("bwd_gate_derivative", "dz[ch * L + t] = dy * yv * sg * (1.0 + zz * (1.0 - sg));",
     "dz[ch * L + t] = dy * yv * sg;"),
    ("bwd_dA_missing_dt", "pA[ch * N + n] += g[n] * hprev * an * dt;", "pA[ch * N + n] += g[n] * hprev * an;"),
    ("bwd_du_missing_skip", "double dut = Dd * dy, ddt = 0.0;", "double dut = 0.0, ddt = 0.0;"),
    ("ssd_sign_of_A", "double a = exp(dt * (double)A[h]);", "double a = exp(-dt * (double)A[h]);"),
    ("ssd_no_dt_on_input", "*s = a * *s + dt * (double)Bt[n] * xt;", "*s = a * *s + (double)Bt[n] * xt;"),
    ("ssd_B_for_C", "acc += (double)Ct[n] * *s;", "acc += (double)Bt[n] * *s;"),
    ("ssd_group_map", "int64_t b = bh / H, h = bh % H, g = h / (H / G);",
     "int64_t b = bh / H, h = bh % H, g = h % G;"),
    ("ssd_drop_D", "double yv = acc + (D ? (double)D[h] * xt : 0.0);", "double yv = acc;"),
    ("conv_update_wrong_weight", "acc += (double)w[d * width + hw] * xt;", "acc += (double)w[d * width] * xt;"),
    ("dir_rows_cols_swapped", "if (order >= 2) return (k % rows) * cols + k / rows;",
     "if (order >= 2) return (k % cols) * rows + k / cols;"),
    ("dir_column_reverse_lost", "if (order == 1 || order == 3) k = L - 1 - k;", "if (order == 1) k = L - 1 - k;"),
    ("zoh_sign", "double bbar = zoh ? (an != 0.0 ? expm1(dt * an) / an : dt) : dt;",
     "double bbar = zoh ? (an != 0.0 ? -expm1(-dt * an) / an : dt) : dt;"),
    ("zoh_zero_A_limit", "double bbar = zoh ? (an != 0.0 ? expm1(dt * an) / an : dt) : dt;",
     "double bbar = zoh ? (an != 0.0 ? expm1(dt * an) / an : 0.0) : dt;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.OracleLib(oracle.compile_source(path, os.path.join(tmp, "libmutant.so")))
        failed = []
        for check in oracle_pins.ALL_CHECKS:
            try:
                check(lib)
            except AssertionError:
                failed.append(check.__name__)
        assert failed, f"no pin catches mutant {name}"
    finally:
        shutil.rmtree(tmp)
