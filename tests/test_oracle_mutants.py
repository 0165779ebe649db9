"""Plants plausible mistakes in copies of the oracle and checks that the pins catch them.

Each mutant is path_oracle.c with one textual change (a dropped term, a wrong sign, a
shifted index, a step in the wrong order), compiled on the CPU into a temporary
library. The pins of test_oracle_pins.py then run against it, and at least one must
fail. The real oracle is restored afterwards.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import build as oracle_build
from tests import test_oracle_pins as pins
from tests import test_bwd_oracle as bpins
from tests import test_producer_oracle as ppins

SRC = oracle_build.SRC

MUTANTS = {
    "transition_sign": ("x[c] -= a * w[c];", "x[c] += a * w[c];"),
    "beta_dropped": ("const double a = beta * dot;", "const double a = dot;"),
    "transition_index_shifted": (
        "apply_transition(x, W + (size_t)j * d, beta[j], d);",
        "apply_transition(x, W + (size_t)(j > 0 ? j - 1 : 0) * d, beta[j > 0 ? j - 1 : 0], d);"),
    "transition_before_score": (
        "        logit[j] = scale * dot + bias;\n        apply_transition(x, W + (size_t)j * d, beta[j], d);",
        "        apply_transition(x, W + (size_t)j * d, beta[j], d);\n"
        "        dot = 0.0;\n        for (int c = 0; c < d; ++c)\n            dot += k_j[c] * x[c];\n"
        "        logit[j] = scale * dot + bias;"),
    "scale_dropped": ("logit[j] = scale * dot + bias;", "logit[j] = dot + bias;"),
    "gate_scaled": ("logit[j] = scale * dot + bias;", "logit[j] = scale * (dot + bias);"),
    "gate_range_includes_j": ("logit[j] = scale * dot + bias;",
                              "logit[j] = scale * dot + bias + (log_f ? log_f[j] : 0.0);"),
    "lse_without_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "softmax_not_normalised": ("const double pj = p[j] / z;", "const double pj = p[j];"),
    "decode_skips_last_key": ("for (int j = 0; j < len; ++j)\n            apply_transition(K",
                              "for (int j = 0; j + 1 < len; ++j)\n            apply_transition(K"),
    "decode_transforms_new_key": (
        "        for (int j = 0; j < len; ++j)\n            apply_transition(K + (size_t)j * d, w_t, beta[h], d);\n"
        "        memcpy(K + (size_t)len * d, k + (size_t)h * d, (size_t)d * sizeof(double));",
        "        memcpy(K + (size_t)len * d, k + (size_t)h * d, (size_t)d * sizeof(double));\n"
        "        for (int j = 0; j <= len; ++j)\n            apply_transition(K + (size_t)j * d, w_t, beta[h], d);"),
    "decode_gate_on_new_key": ("cb[len] = 0.0;", "cb[len] = log_f[h];"),
    # w / beta producer
    "producer_conv_forward_in_time": (
        "acc += conv[(size_t)ch * 3 + 1] * y[(size_t)(t - 1) * C + ch];",
        "acc += conv[(size_t)ch * 3 + 1] * y[(size_t)(t + 1 < L ? t + 1 : t) * C + ch];"),
    "producer_taps_reversed": (
        "double acc = conv[(size_t)ch * 3 + 2] * y[(size_t)t * C + ch];",
        "double acc = conv[(size_t)ch * 3 + 0] * y[(size_t)t * C + ch];"),
    "producer_norm_over_all_heads": (
        "for (int c = 0; c < d; ++c)\n                    ss += yc[h * d + c] * yc[h * d + c];",
        "for (int c = 0; c < C; ++c)\n                    ss += yc[c] * yc[c];"),
    "producer_beta_without_factor_2": ("double be = 2.0 / (1.0 + exp(-a));",
                                       "double be = 1.0 / (1.0 + exp(-a));"),
    "producer_beta_not_clipped": ("if (be > beta_max)\n                    be = beta_max;",
                                  "(void)beta_max;"),
    "producer_projects_previous_token": (
        "acc += w_down[(size_t)r * D + c] * xb[(size_t)t * D + c];",
        "acc += w_down[(size_t)r * D + c] * xb[(size_t)(t > 0 ? t - 1 : 0) * D + c];"),
    # backward
    "bwd_dS_without_row_term": ("const double dS = p[j] * (logit[j] - Dsum);",
                                "const double dS = p[j] * logit[j];"),
    "bwd_dk_unscaled": ("dK[(size_t)j * d + c] += scale * dS * x_j[c];",
                        "dK[(size_t)j * d + c] += dS * x_j[c];"),
    "bwd_dw_drops_term": ("dW[(size_t)(j + 1) * d + c] -= b * (wu * g[c] + wg * u[c]);",
                          "dW[(size_t)(j + 1) * d + c] -= b * (wu * g[c]);"),
    "bwd_gradient_not_transported": ("g[c] -= b * wg * w[c];", "g[c] -= 0.0 * wg * w[c];"),
    "bwd_dbeta_sign": ("dbeta[j + 1] -= wg * wu;", "dbeta[j + 1] += wg * wu;"),
    "bwd_gate_index_shifted": ("dlogf[j + 1] += gate_acc;", "dlogf[j] += gate_acc;"),
}


def run_all_pins():
    """Runs every pin; returns the names of those that failed."""
    failed = []
    checks = [
        ("hand", pins.test_hand_example_logits_outputs_and_fox, ()),
        ("beta0", pins.test_beta_zero_is_causal_softmax_attention, (37, 8)),
        ("diag", pins.test_diagonal_logit_is_plain_dot_product, ()),
        ("brute", pins.test_brute_force_explicit_matrices, (9, 8)),
        ("repeat", pins.test_repeated_transition_closed_form, ()),
        ("norm", pins.test_reflections_preserve_norm_and_general_beta_contracts, ()),
        ("order", pins.test_order_of_transitions_matters, ()),
        ("fox", pins.test_fox_reductions, ()),
        ("decode", pins.test_decode_from_empty_cache_matches_prefill, (False,)),
        ("decode_fox", pins.test_decode_from_empty_cache_matches_prefill, (True,)),
        ("rows", pins.test_sampled_rows_match_full_forward, ()),
        ("p_hand", ppins.test_hand_example, ()),
        ("p_rank1", ppins.test_rank_one_equal_taps_closed_form, ()),
        ("p_reach", ppins.test_convolution_reaches_two_tokens_back_and_no_further, ()),
        ("p_shift", ppins.test_lag_one_tap_shifts_the_output_by_one_token, ()),
        ("p_norm", ppins.test_unit_norm_scale_invariance_and_heads_independent, ()),
        ("p_beta", ppins.test_beta_limits, ()),
        ("b_fd", bpins.test_bwd_matches_finite_differences, (False,)),
        ("b_fd_fox", bpins.test_bwd_matches_finite_differences, (True,)),
        ("b_beta0", bpins.test_bwd_beta_zero_closed_form, ()),
        ("b_sign", bpins.test_bwd_sign_of_w, ()),
        ("b_dv", bpins.test_bwd_dv_is_p_transpose_dout, ()),
    ]
    for name, fn, args in checks:
        try:
            with np.errstate(all="ignore"):
                fn(*args)
        except AssertionError:
            failed.append(name)
    return failed


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation site not found exactly once"
    src = os.path.join(mutant_dir, name + ".c")
    lib = os.path.join(mutant_dir, "lib" + name + ".so")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", src, "-o", lib,
                    "-lm"], check=True)
    prev = oracle.swap_library(lib)
    try:
        failed = run_all_pins()
    finally:
        oracle.restore_library(prev)
    assert failed, "no pin caught mutant %s" % name


def test_unmutated_oracle_passes_every_pin():
    assert run_all_pins() == []
