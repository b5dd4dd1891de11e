"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins catch every one of them."""
import pytest

import oracle
from oracle_pins import PINS

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("no_decay", "S[(size_t)i * d + j] *= a[i];", "S[(size_t)i * d + j] *= 1.0;"),
    ("decay_on_columns", "S[(size_t)i * d + j] *= a[i];", "S[(size_t)i * d + j] *= a[j];"),
    ("decay_sign", "gkv[c] = -exp(", "gkv[c] = exp("),
    ("no_beta_on_erase", "-beta * kv[i] * u[j]", "-kv[i] * u[j]"),
    ("no_erase", "-beta * kv[i] * u[j]", "0.0"),
    ("readout_transposed", "s += S[(size_t)i * d + j] * qv[i];", "s += S[(size_t)j * d + i] * qv[i];"),
    ("taps_reversed", "w[0] * x_m3 + w[1] * x_m2 + w[2] * x_m1 + w[3] * x_t[c]",
     "w[3] * x_m3 + w[2] * x_m2 + w[1] * x_m1 + w[0] * x_t[c]"),
    ("no_silu", "y[c] = silu(pre);", "y[c] = pre;"),
    ("k_not_normalised", "l2_normalize(kv, d, J->l2_eps);", ""),
    ("window_not_shifted", "win[2 * HD3 + ch] = x_t[c];", "win[2 * HD3 + ch] = x_m1;"),
    ("rms_sum_not_mean", "ms /= d;", ""),
    ("no_gate", "* inv_rms *\n                            sigmoid(J->gate_logit[row + j]);", "* inv_rms;"),
    ("erase_uses_q", "s += kv[i] * S[(size_t)i * d + j];", "s += qv[i] * S[(size_t)i * d + j];"),
    ("write_uses_q", "beta * kv[i] * vv[j]", "beta * qv[i] * vv[j]"),
    ("no_softplus", "softplus(J->z[row + c] + J->dt_bias[(size_t)h * d + c])",
     "(J->z[row + c] + J->dt_bias[(size_t)h * d + c])"),
    ("no_dt_bias", " + J->dt_bias[(size_t)h * d + c]", ""),
    ("no_gamma", "J->gamma[(size_t)h * d + j] * op[j]", "op[j]"),
    ("beta_not_squashed", "sigmoid(J->beta_logit[bth])", "(J->beta_logit[bth])"),
    ("l2_eps_dropped", "1.0 / sqrt(ss + eps)", "1.0 / sqrt(ss)"),
    ("rms_eps_dropped", "sqrt(ms + J->rms_eps)", "sqrt(ms)"),
    ("exp_alog_dropped", "-exp(J->A_log[(size_t)h * d + c])", "-(J->A_log[(size_t)h * d + c])"),
    # low-rank front-end
    ("lowrank_fa_transposed", "W_fa[(size_t)r * hidden + j] * xn[j]", "W_fa[(size_t)j * rank + r] * xn[j]"),
    ("lowrank_fb_transposed", "W_fb[m * rank + r] * u[r]", "W_fb[(size_t)r * HD + m] * u[r]"),
    ("lowrank_skips_fa", "W_fb[m * rank + r] * u[r]", "W_fb[m * rank + r] * xn[r]"),
    ("lowrank_beta_from_fa", "W_bp[(size_t)h * hidden + j] * xn[j]", "W_fa[(size_t)h * hidden + j] * xn[j]"),
    ("lowrank_token_stride", "const double *xn = x + (size_t)n * hidden;", "const double *xn = x + (size_t)n * rank;"),
    ("lowrank_head_offset", "z[(size_t)n * HD + m] = s;", "z[(size_t)n * HD + (m + d) % HD] = s;"),
    # projections
    ("project_transposed", "s += wi[j] * xn[j];", "s += W[(size_t)j * out + i] * xn[j];"),
    ("project_token_stride", "const double *xn = x + (size_t)n * in;", "const double *xn = x + (size_t)n * out;"),
    ("project_output_shifted", "y[(size_t)n * out + i] = s;", "y[(size_t)n * out + (i + 1) % out] = s;"),
    # bfloat16 state storage
    ("bf16_ties_away", "const double r = nearbyint(m);", "const double r = round(m);"),
    ("bf16_truncates", "const double r = nearbyint(m);", "const double r = trunc(m);"),
    ("bf16_no_subnormal_spacing", "if (E < -126) E = -126;", ""),
    ("bf16_state_not_rounded", "if (J->state_bf16)\n", "if (0)\n"),
    ("bf16_rounds_before_readout", "/* \"O projection\" without the W_o / W_g matmuls: o_pre = S^T q. */",
     "if (J->state_bf16) for (size_t i = 0; i < (size_t)d * d; ++i)\n"
     "            S[i] = kda_oracle_bf16_value(kda_oracle_bf16_round(S[i]));"),
]


def _fails(lib):
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    lib = oracle.build_variant(src.replace(old, new), name)
    assert _fails(lib), f"no pin catches the planted mistake {name}"
