"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutation is a plausible slip (a flipped tie rule, an off-by-one capacity
test, a swapped threshold, a dropped term, a transposed operand, the sample
instead of the population variance, ...). The copy is compiled on the CPU into
a temporary library; the real oracle is untouched.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTATIONS = {
    "tie_rule_higher_index_wins": ("h[e] > h[best]", "h[e] >= h[best]"),
    "capacity_test_inclusive": ("(p < C)", "(p <= C)"),
    "capacity_ceil": ("floor((double)k", "ceil((double)k"),
    "count_only_kept": ("count[e] = p + 1;", "count[e] = p + (p < C);"),
    "threshold_swapped": ("chosen >= 0 ? hk1[t] : hk[t]", "chosen >= 0 ? hk[t] : hk1[t]"),
    "load_sign": ("(c[(size_t)t * E + e] - thr) / s", "(thr - c[(size_t)t * E + e]) / s"),
    "router_bias_dropped": ("if (bias) acc += (double)bias[e];", ""),
    "noise_unscaled": ("h = acc + (double)noise[(size_t)t * E + e] * s;",
                       "h = acc + (double)noise[(size_t)t * E + e];"),
    "softplus_as_log_exp": ("log1p(exp(-fabs(z)))", "log(exp(-fabs(z)))"),
    "relu_dropped": ("if (h[f] < 0.0) h[f] = 0.0;", ""),
    "gate_not_applied": ("yt[c] += g * oc;", "yt[c] += oc;"),
    "w1_transposed": ("size_t row = ((size_t)e * d + i) * d_ff;\n        for (int f = 0; f < d_ff; ++f) h[f] += xi * orc_in(W1, w_dtype, row + f);",
                      "for (int f = 0; f < d_ff; ++f) h[f] += xi * orc_in(W1, w_dtype, ((size_t)e * d_ff + f) * d + i);"),
    "b2_outside_gate": ("double oc = o[c] + (b2 ? orc_in(b2, w_dtype, (size_t)e * d + c) : 0.0);\n        yt[c] += g * oc;",
                        "double oc = o[c];\n        yt[c] += g * oc + (b2 ? orc_in(b2, w_dtype, (size_t)e * d + c) : 0.0);"),
    "sample_variance": ("var /= n;", "var /= (n - 1);"),
    "cv_not_squared": ("return var / (mean * mean);", "return sqrt(var) / mean;"),
    "switch_gate_renormalised": ("gate[(size_t)t * k] = exp(h[order[0]] - top) / z;\n    } else {",
                                 "gate[(size_t)t * k] = 1.0;\n    } else {"),
    "switch_aux_no_E": ("out3[2] = 0.01 * (double)E * sfp;", "out3[2] = 0.01 * sfp;"),
    "importance_first_choice_only": ("if (chosen >= 0) imp += gate[(size_t)t * k + chosen];",
                                     "if (chosen == 0) imp += gate[(size_t)t * k + chosen];"),
    "kplus1_threshold_off_by_one": ("hk1[t] = (k < E) ? h[order[k]] : -INFINITY;",
                                    "hk1[t] = (k < E) ? h[order[k - 1]] : -INFINITY;"),
    "phi_argument_unscaled": ("erfc(-u / sqrt(2.0))", "erfc(-u)"),
    "hier_gate_not_product": ("gate[(size_t)t * k + q * ks + r] = g_p[(size_t)t * kp + q] * sg[r];",
                              "gate[(size_t)t * k + q * ks + r] = sg[r];"),
    "hier_index_not_offset": ("idx[(size_t)t * k + q * ks + r] = i * b + sidx[r];",
                              "idx[(size_t)t * k + q * ks + r] = sidx[r];"),
    "hier_guard_missing": ("count[i] > 0 ? load_p[i] * loadsec[e] / (double)count[i] : 0.0",
                           "load_p[i] * loadsec[e] / (double)count[i]"),
    "hier_load_not_normalised": ("count[i] > 0 ? load_p[i] * loadsec[e] / (double)count[i] : 0.0",
                                 "count[i] > 0 ? load_p[i] * loadsec[e] : 0.0"),
    "hier_primary_load_dropped": ("count[i] > 0 ? load_p[i] * loadsec[e] / (double)count[i] : 0.0",
                                  "count[i] > 0 ? loadsec[e] / (double)count[i] : 0.0"),
    "hier_threshold_swapped": ("chosen ? hk1s[(size_t)t * kp + q] : hks[(size_t)t * kp + q]",
                               "chosen ? hks[(size_t)t * kp + q] : hk1s[(size_t)t * kp + q]"),
    "bal_tie_higher_token_wins": ("if (best < 0 || P[(size_t)t * E + i] > P[(size_t)best * E + i]) best = t;",
                                  "if (best < 0 || P[(size_t)t * E + i] >= P[(size_t)best * E + i]) best = t;"),
    "bal_gate_not_renormalised": ("mask[(size_t)t * E + i] ? P[(size_t)t * E + i] / z : 0.0;",
                                  "mask[(size_t)t * E + i] ? P[(size_t)t * E + i] : 0.0;"),
    "bal_threshold_inclusive": ("mask[u] = P[u] > (double)thr[u % E] ? 1 : 0;",
                                "mask[u] = P[u] >= (double)thr[u % E] ? 1 : 0;"),
    "bal_loss_sign": ("s += (mt - (double)mask_batch[(size_t)t * E + i]) * (x - th);",
                      "s += ((double)mask_batch[(size_t)t * E + i] - mt) * (x - th);"),
    "bal_rows_rounded_up": ("long long m = (long long)k * T / E;",
                            "long long m = ((long long)k * T + E - 1) / E;"),
    "softmax_no_max_shift": ("for (int e = 0; e < E; ++e) z += exp(h[e] - mx);\n    for (int e = 0; e < E; ++e) P[(size_t)t * E + e] = exp(h[e] - mx) / z;",
                             "for (int e = 0; e < E; ++e) z += exp(h[e]);\n    for (int e = 0; e < E; ++e) P[(size_t)t * E + e] = exp(h[e]) / z;"),
    "hier_secondary_load_dropped": ("      count[i] += 1;\n      for (int j = 0; j < b; ++j) {",
                                       "      count[i] += 1;\n      for (int j = 0; j < b && 0; ++j) {"),
    "bwd_residual_dropped": ("for (int i = 0; i < d; ++i) dx[(size_t)t * d + i] += dy[(size_t)t * d + i];", ""),
    "bwd_relu_mask_dropped": ("dpre[f] = pre[f] > 0.0 ? dh : 0.0;", "dpre[f] = dh;"),
    "bwd_dropped_choices_trained": ("if (!keep[(size_t)t * k + j]) continue;\n      const int e = idx[(size_t)t * k + j];\n      const double g",
                                    "const int e = idx[(size_t)t * k + j];\n      const double g"),
    "bwd_w2_transposed": ("dh += orc_in(W2, w_dtype, ((size_t)e * d_ff + f) * d + cc) * du;",
                          "dh += orc_in(W2, w_dtype, ((size_t)e * d + cc) * d_ff + f) * du;"),
    "bwd_softmax_jacobian_sign": ("gate[(size_t)t * k + j] * (dG[j] - sum);",
                                  "gate[(size_t)t * k + j] * (dG[j] + sum);"),
    "bwd_threshold_owner_dropped": ("dH[(size_t)t * E + owner] -= g;", ""),
    "bwd_cv2_mean_term_dropped": (" - 2.0 * var / (E * m * m * m));", ");"),
    "bwd_softplus_slope_dropped": ("dsg[u] / (1.0 + exp(-zn[u]))", "dsg[u]"),
    "bwd_noise_scale_dropped": ("dsg[u] += (double)noise[u] * dH[u];", "dsg[u] += dH[u];"),
    "bwd_aux_not_averaged": ("w_aux * 0.01 * E * f[e] / T;", "w_aux * 0.01 * E * f[e];"),
    "bwd_importance_only_kept": ("dG[j] = dg[(size_t)t * k + j] + dimp[idx[(size_t)t * k + j]];",
                                 "dG[j] = dg[(size_t)t * k + j] + (dg[(size_t)t * k + j] != 0.0 ? dimp[idx[(size_t)t * k + j]] : 0.0);"),
    "hbwd_primary_share_unweighted": ("dgp[q] += dprod * sg[r];", "dgp[q] += dprod;"),
    "hbwd_secondary_share_unweighted": ("dsg[r] = dprod * gp;", "dsg[r] = dprod;"),
    "hbwd_group_load_not_normalised": ("dloadsec[e] = dloadH[e] * load_p[i] / (double)gcount[i];",
                                       "dloadsec[e] = dloadH[e] * load_p[i];"),
    "hbwd_primary_load_dropped": ("dload_p[i] += dloadH[e] * loadsec[e] / (double)gcount[i];", ""),
    "hbwd_group_owner_not_offset": ("orc_next_unchosen(hs, b, picks, ks, i * b)",
                                    "orc_next_unchosen(hs, b, picks, ks, 0)"),
    "balbwd_renormalisation_ignored": ("dP[i] = mask[(size_t)t * E + i] ? (dG[(size_t)t * E + i] - gd) / S : 0.0;",
                                       "dP[i] = mask[(size_t)t * E + i] ? dG[(size_t)t * E + i] : 0.0;"),
    "balbwd_loss_sign": ("dP[i] += w_bal * ((p[i] > (double)thr[i] ? 1.0 : 0.0) - (double)mb[(size_t)t * E + i]);",
                         "dP[i] += w_bal * ((double)mb[(size_t)t * E + i] - (p[i] > (double)thr[i] ? 1.0 : 0.0));"),
    "balbwd_softmax_mean_dropped": ("dH[(size_t)t * E + i] = p[i] * (dP[i] - pd);",
                                    "dH[(size_t)t * E + i] = p[i] * dP[i];"),
    "load_uses_noisy_logit": ("p = orc_phi((c[(size_t)t * E + e] - thr) / s);",
                              "p = orc_phi((H[(size_t)t * E + e] - thr) / s);"),
    "capacity_without_k": ("double raw = floor((double)k * (double)T * cf / (double)E);",
                           "double raw = floor((double)T * cf / (double)E);"),
    "slot_position_inclusive": ("pos[(size_t)t * k + j] = p;", "pos[(size_t)t * k + j] = p + 1;"),
    "residual_dropped": ("for (int i = 0; i < d; ++i) yt[i] = orc_in(x, x_dtype, (size_t)t * d + i);",
                         "for (int i = 0; i < d; ++i) yt[i] = 0.0;"),
    "cv2_over_mean": ("return var / (mean * mean);", "return var / mean;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "moe_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    mutant = oracle.variant(str(mutated), str(tmp_path))
    caught = None
    for pin in ALL_PINS:  # one failing pin is enough
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            caught = pin.__name__
            break
    assert caught, f"no pin caught the planted mistake {name}"
