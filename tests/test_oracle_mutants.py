"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/moe_oracle.c, builds
it with the oracle's own flags, and runs the pin suite (tests/test_oracle_pins.py)
against that library in a child process.  The case passes when the pins named
beside the mistake fail, so that every pinned branch of the oracle is shown to
be held by some pin and not by the oracle's agreement with itself.  Mistakes
that are provably harmless (walking a token's preference order from position 0
instead of r: every earlier position is held or full) are not listed.
"""
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
PINS = os.path.join(HERE, "test_oracle_pins.py")

# name -> (edits (old, new), each `old` occurring exactly once, pins that must fail)
MUTANTS = {
    # capacity and routing ([coreui] §5.2 capacity; [mhpn] §2.3 penalty; top-k order)
    "capacity_floor": ([("return (num + den - 1) / den;", "return num / den;")],
                       ["test_capacity_page_value"]),
    "ties_to_higher_index": ([("    return a < b;\n}", "    return a > b;\n}")],
                             ["test_preference_matches_sorted_with_ties", "test_equal_logits_pick_lowest_indices"]),
    "penalty_sign": ([("s[e] = zt - pen;", "s[e] = zt + pen;")], ["test_penalty_is_two_rounded_fp32_ops"]),
    "penalty_fused": ([("volatile float pen = lambda * usage[e];\n                s[e] = zt - pen;",
                        "s[e] = fmaf(-lambda, usage[e], zt);")], ["test_penalty_is_two_rounded_fp32_ops"]),
    "temperature_after_penalty": ([("s[e] = zt - pen;", "s[e] = (z[e] - pen) / tau;")],
                                  ["test_temperature_comes_before_the_penalty"]),
    "P_not_averaged": ([("P[e] = T > 0 ? (float)(psum[e] / (double)T) : 0.0f;",
                         "P[e] = T > 0 ? (float)(psum[e]) : 0.0f;")], ["test_softmax_and_stats_match_scipy"]),
    "P_of_topk_only": ([("for (int e = 0; e < E; ++e) psum[e] += p[e];",
                         "for (int r = 0; r < k; ++r) psum[order[r]] += p[order[r]];")],
                       ["test_softmax_and_stats_match_scipy"]),
    "f_not_over_T": ([("f[e] = T > 0 ? (float)((double)counts_pre[e] / (double)T) : 0.0f;",
                       "f[e] = T > 0 ? (float)counts_pre[e] : 0.0f;")], ["test_softmax_and_stats_match_scipy"]),
    "softmax_of_logits": ([("softmax_row(E, s, p);", "softmax_row(E, z, p);")],
                          ["test_softmax_and_stats_match_scipy", "test_temperature_sharpens_softmax"]),
    # router front end ([2kiu] §5.2 normalisation; [cnnetsun] §3.1 two-layer router)
    "layernorm_unbiased_variance": ([("var /= (double)d;", "var /= (double)(d - 1);")],
                                    ["test_layernorm_worked_example", "test_layernorm_router_reduces_to_torch"]),
    "layernorm_eps_outside_sqrt": ([("1.0 / sqrt(var + (double)eps)", "1.0 / (sqrt(var) + (double)eps)")],
                                   ["test_layernorm_router_reduces_to_torch"]),
    "l2_eps_added": ([("if (nrm < (double)eps) nrm = (double)eps;", "nrm += (double)eps;")],
                     ["test_l2_norm_eps_is_a_floor"]),
    "router_hidden_no_silu": ([("a[j] = u / (1.0 + exp(-u));", "a[j] = u;")],
                              ["test_two_layer_router_identity_is_silu", "test_two_layer_router_reduces_to_torch"]),
    "capacity_override_ignored": ([("if (explicit_cap > 0) return explicit_cap;", "(void)explicit_cap;")],
                                  ["test_capacity_explicit_override"]),
    "logits_bias_dropped": ([("                if (bias) acc += (double)bias[e];\n                z[e] = (float)acc;",
                              "                z[e] = (float)acc;")], ["test_logits_match_float64_matmul"]),
    "temperature_multiplies": ([("volatile float zt = z[e] / tau;", "volatile float zt = z[e] * tau;")],
                               ["test_temperature_comes_before_the_penalty", "test_temperature_sharpens_softmax"]),
    "nan_not_rejected": ([("if (isnan(s_row[e])) return 5;", "(void)0;")], ["test_nan_score_is_an_error"]),
    "softmax_inf_limit_uniform": ([("p[e] = ((double)s[e] == m) ? 1.0 / n : 0.0;", "p[e] = 1.0 / E;")],
                                  ["test_softmax_limits"]),
    "layernorm_gamma_beta_swapped": ([("(gamma ? (double)gamma[i] : 1.0) + (beta ? (double)beta[i] : 0.0)",
                                       "(beta ? (double)beta[i] : 1.0) + (gamma ? (double)gamma[i] : 0.0)")],
                                     ["test_layernorm_worked_example", "test_layernorm_router_reduces_to_torch"]),
    # dispatch ([mhpn] §2.3 the 128th token; rank-major order; capacity cap)
    "rank_minor_order": ([("for (int r = 0; r < k; ++r) {\n            for (int t = 0; t < T; ++t) {",
                           "for (int t = 0; t < T; ++t) {\n            for (int r = 0; r < k; ++r) {")],
                         ["test_worked_case_128_identical_tokens", "test_rank_major_order_matters"]),
    "fill_past_capacity": ([("if (fill[e] >= C) continue;", "if (fill[e] > C) continue;")],
                           ["test_page_overflow_case", "test_drop_case"]),
    "no_held_check": ([("if (held) continue;", "(void)held;")], ["test_dispatch_brute_force_tiny"]),
    "weights_not_renormalised": ([("(float)(p[e] / tot)", "(float)(p[e])")],
                                 ["test_k1_weight_is_one", "test_reroute_weight_uses_the_expert_actually_used"]),
    "reroute_weight_of_first_pick": ([("(float)(p[e] / tot)", "(float)(p[order[(size_t)t * E + r]] / tot)")],
                                     ["test_reroute_weight_uses_the_expert_actually_used"]),
    "reroute_flag_against_rank0": ([("flags[idx] = (chosen != pi[r]) ? 1 : 0;",
                                     "flags[idx] = (chosen != pi[0]) ? 1 : 0;")],
                                   ["test_dispatch_invariants_random"]),
    "perm_holds_token": ([("perm[offsets[assign[idx]] + slot[idx]] = (int32_t)idx;",
                           "perm[offsets[assign[idx]] + slot[idx]] = (int32_t)t;")],
                         ["test_dispatch_invariants_random"]),
    "drop_flag_value": ([("flags[idx] = 2;", "flags[idx] = 3;")], ["test_drop_case"]),
    "reroutes_counted_for_every_pick": ([("nre += (chosen != pi[r]);", "nre += 1;")],
                                        ["test_worked_case_128_identical_tokens", "test_page_overflow_case"]),
    # experts ([mhpn] §3.1 SwiGLU W1 gate, W3 up)
    "gate_up_swapped": ([("a[j] = silu(g) * u;", "a[j] = silu(u) * g;")],
                        ["test_gate_and_up_branches_are_not_swapped"]),
    "silu_sign": ([("static double silu(double x) { return x / (1.0 + exp(-x)); }",
                    "static double silu(double x) { return x / (1.0 + exp(x)); }")],
                  ["test_dense_swiglu_reduces_to_torch"]),
    # e4m3 format and the FP8 expert path ([2kiu] §5.1 quantised experts)
    "e4m3_subnormal_step": ([("double q = a / ldexp(1.0, -9);", "double q = a / ldexp(1.0, -10);")],
                            ["test_e4m3_encode_matches_torch", "test_e4m3_encode_inverts_decode"]),
    "e4m3_saturates_to_nan": ([("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;")],
                              ["test_e4m3_encode_ties_and_saturation"]),
    "e4m3_nan_encodes_as_zero": ([("if (isnan(v)) return 0x7F;", "if (isnan(v)) return 0;")],
                                 ["test_e4m3_nan_codes"]),
    "q8_zero_row_scale_0": ([("const float s = amax > 0.0f ? amax / 448.0f : 1.0f;", "const float s = amax / 448.0f;")],
                            ["test_quantize_row_matches_torch"]),
    "e4m3_ties_away": ([("double m = (q - f > 0.5 || (q - f == 0.5 && fmod(f, 2.0) != 0.0)) ? f + 1.0 : f;\n"
                         "    if (m == 8.0)",
                         "double m = (q - f >= 0.5) ? f + 1.0 : f;\n    if (m == 8.0)")],
                       ["test_e4m3_encode_ties_and_saturation", "test_q8_activation_rounding_hand_case"]),
    "quant_scale_not_448": ([("amax / 448.0f", "amax / 256.0f")],
                            ["test_quantize_row_matches_torch", "test_q8_activation_quantisation_is_identity_on_exact_rows"]),
    "weight_scale_of_row_0": ([("return e4m3_tab[w->q[r * w->cols + c]] * (double)w->s[r];",
                                "return e4m3_tab[w->q[r * w->cols + c]] * (double)w->s[0];")],
                              ["test_q8_experts_equal_bf16_experts_on_exact_weights"]),
    "token_dequant_drops_scale": ([("xf[i] = oracle_e4m3_value(codes[i]) * (double)sc;",
                                    "xf[i] = oracle_e4m3_value(codes[i]);")],
                                  ["test_q8_activation_quantisation_is_identity_on_exact_rows",
                                   "test_q8_activation_rounding_hand_case"]),
    "token_rows_not_quantised": ([("for (int i = 0; i < d; ++i) xf[i] = oracle_e4m3_value(codes[i]) * (double)sc;",
                                   "(void)0;")], ["test_q8_activation_rounding_hand_case"]),
    "act_not_rounded_to_bf16": ([("tmp[j] = bf16_to_f32(f32_to_bf16_rne((float)a[j]));\n        oracle_quantize_row(",
                                  "tmp[j] = (float)a[j];\n        oracle_quantize_row(")],
                                ["test_q8_activation_rounding_hand_case"]),
    "act_scale_of_token_row": ([("oracle_quantize_row(F, tmp, codes, &sc);",
                                 "for (int j = 0; j < F; ++j) codes[j] = oracle_e4m3_encode(tmp[j] / sc);")],
                               ["test_q8_activation_quantisation_is_identity_on_exact_rows",
                                "test_q8_activation_rounding_hand_case"]),
    "act_max_before_swiglu": ([("        a[j] = silu(g) * u;\n    }",
                                "        a[j] = silu(g) * u;\n        if (fabs(g) > gmax) gmax = fabs(g);\n    }"),
                               ("malloc((size_t)(d > F ? d : F));\n    float sc = 1.0f;\n",
                                "malloc((size_t)(d > F ? d : F));\n    float sc = 1.0f;\n    double gmax = 0.0;\n"),
                               ("oracle_quantize_row(F, tmp, codes, &sc);",
                                "sc = gmax > 0.0 ? (float)gmax / 448.0f : 1.0f; "
                                "for (int j = 0; j < F; ++j) codes[j] = oracle_e4m3_encode(tmp[j] / sc);")],
                              ["test_q8_activation_quantisation_is_identity_on_exact_rows",
                               "test_q8_activation_rounding_hand_case"]),
    # NVFP4: e2m1 elements with e4m3 scales per 16 and a row scale ([2kiu] §5.1 4-bit experts)
    "e2m1_ties_away": ([("if (dd < bd || (dd == bd && (c & 1) == 0 && (best & 1) == 1))", "if (dd <= bd)")],
                       ["test_e2m1_encode_is_nearest_with_ties_to_even", "test_q4_activation_quantisation_hand_case"]),
    "e2m1_subnormal_doubled": ([("const double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);",
                                 "const double v = (e == 0) ? 1.0 * m : ldexp(1.0 + 0.5 * m, e - 1);")],
                               ["test_e2m1_all_codes"]),
    "nvfp4_zero_row_scale_0": ([("const float s = amax > 0.0f ? amax / 2688.0f : 1.0f;", "const float s = amax / 2688.0f;")],
                               ["test_nvfp4_zero_row_and_underflowing_block"]),
    "nvfp4_zero_divisor_saturates": ([("const uint8_t c = den > 0.0f ? oracle_e2m1_encode(x[i] / den) : 0;",
                                       "const uint8_t c = oracle_e2m1_encode(x[i] / den);")],
                                     ["test_nvfp4_zero_row_and_underflowing_block"]),
    "nvfp4_scale_448": ([("amax / 2688.0f", "amax / 448.0f")],
                        ["test_nvfp4_row_quantisation_is_exact_on_representable_rows",
                         "test_nvfp4_row_quantisation_hand_case"]),
    "nvfp4_block_scale_not_over_6": ([("const float u = t / 6.0f;", "const float u = t;")],
                                     ["test_nvfp4_row_quantisation_is_exact_on_representable_rows",
                                      "test_nvfp4_row_quantisation_hand_case"]),
    "nvfp4_nibbles_swapped": ([("codes[i / 2] |= (uint8_t)(c << (4 * (i & 1)));",
                                "codes[i / 2] |= (uint8_t)(c << (4 * (1 - (i & 1))));")],
                              ["test_nvfp4_row_quantisation_is_exact_on_representable_rows",
                               "test_nvfp4_row_quantisation_hand_case"]),
    "q4_weight_blocks_of_32": ([("w->bs[(r * w->cols + c) / 16]", "w->bs[(r * w->cols + c) / 32]")],
                               ["test_q4_experts_equal_bf16_experts_on_exact_weights"]),
    "q4_act_not_rounded_to_bf16": ([("tmp[j] = bf16_to_f32(f32_to_bf16_rne((float)a[j]));\n        nvfp4_row(",
                                     "tmp[j] = (float)a[j];\n        nvfp4_row(")],
                                   ["test_q4_activation_quantisation_hand_case"]),
    "q4_token_rows_not_quantised": ([("nvfp4_row(d, tmp, xf);", "(void)0;")],
                                    ["test_q4_activation_quantisation_hand_case"]),
    "q4_weight_row_scale_dropped": ([("e2m1_tab[code] * e4m3_tab[w->bs[(r * w->cols + c) / 16]] * (double)w->s[r];",
                                      "e2m1_tab[code] * e4m3_tab[w->bs[(r * w->cols + c) / 16]];")],
                                    ["test_q4_experts_equal_bf16_experts_on_exact_weights"]),
    "q4_act_blocks_of_32": ([("oracle_e4m3_value(bs[i / 16])", "oracle_e4m3_value(bs[i / 32])")],
                            ["test_q4_activation_quantisation_hand_case"]),
    # backward with the routing held fixed ([cnnetsun] §4.2 aux loss; [coreui] §3.1)
    "bwd_dsilu_drops_term": ([("sg * (1.0 + g[j] * (1.0 - sg))", "sg")],
                             ["test_backward_dense_swiglu_is_torch_autograd"]),
    "bwd_dh_misses_up_branch": ([("(double)bf16_to_f32(W1[(size_t)j * d + i]) * dg +\n"
                                  "                                             (double)bf16_to_f32(W3[(size_t)j * d + i]) * du;",
                                  "(double)bf16_to_f32(W1[(size_t)j * d + i]) * dg;")],
                                ["test_backward_dense_swiglu_is_torch_autograd"]),
    "bwd_dy_without_weight": ([("dy[c] = cw[r] * (double)gt[c];", "dy[c] = (double)gt[c];")],
                              ["test_backward_matches_torch_autograd"]),
    "bwd_dw2_of_gate": ([("DW2[(size_t)c * F + j] += dy[c] * a[j];", "DW2[(size_t)c * F + j] += dy[c] * g[j];")],
                        ["test_backward_dense_swiglu_is_torch_autograd"]),
    "bwd_dw1_dw3_swapped": ([("DW1[(size_t)j * d + i] += dg * x[i];\n                    DW3[(size_t)j * d + i] += du * x[i];",
                              "DW1[(size_t)j * d + i] += du * x[i];\n                    DW3[(size_t)j * d + i] += dg * x[i];")],
                            ["test_backward_dense_swiglu_is_torch_autograd"]),
    "bwd_renorm_mean_dropped": ([("dp[e] += (dcw[r] - m) / S;", "dp[e] += dcw[r] / S;")],
                                ["test_backward_matches_torch_autograd"]),
    "bwd_tau_dropped": ([("const double dz = p[e] * (dp[e] - pd) / (double)tau;",
                          "const double dz = p[e] * (dp[e] - pd);")], ["test_backward_matches_torch_autograd"]),
    "bwd_dP_not_over_T": ([("dp[e] = dP ? (double)dP[e] / (double)T : 0.0;", "dp[e] = dP ? (double)dP[e] : 0.0;")],
                          ["test_backward_dropped_token_gets_only_the_aux_gradient"]),
    "bwd_dh_misses_router": ([("dh[(size_t)t * d + i] += dz * (double)bf16_to_f32(we[i]);", "(void)we;")],
                             ["test_backward_matches_torch_autograd"]),
    # further branches: router biases and β, the L2 norm, statistics per rank, the combine
    # weights, the slot's token, the quantisers' maxima, the backward's router-side terms
    "router_linear_bias_dropped": ([("for (int i = 0; i < d; ++i) acc += x[i] * (double)bf16_to_f32(we[i]);\n"
                                    "                if (bias) acc += (double)bias[e];",
                                    "for (int i = 0; i < d; ++i) acc += x[i] * (double)bf16_to_f32(we[i]);")],
                                   ["test_layernorm_router_reduces_to_torch"]),
    "router_hidden_bias_dropped": ([("for (int j = 0; j < hidden; ++j) acc += a[j] * (double)bf16_to_f32(we[j]);\n"
                                    "                if (bias) acc += (double)bias[e];",
                                    "for (int j = 0; j < hidden; ++j) acc += a[j] * (double)bf16_to_f32(we[j]);")],
                                   ["test_two_layer_router_orientation"]),
    "layernorm_beta_dropped": ([(" + (beta ? (double)beta[i] : 0.0)", "")],
                               ["test_layernorm_worked_example", "test_layernorm_router_reduces_to_torch"]),
    "l2_norm_not_rooted": ([("double nrm = sqrt(ss);", "double nrm = ss;")],
                           ["test_l2_norm_worked_example_and_torch", "test_l2_norm_eps_is_a_floor"]),
    "counts_pre_of_rank0": ([("counts_pre[order[r]] += 1;", "counts_pre[order[0]] += 1;")],
                            ["test_softmax_and_stats_match_scipy"]),
    "topk_p_of_rank0": ([("topk_p[(size_t)t * k + r] = (float)p[order[r]];",
                          "topk_p[(size_t)t * k + r] = (float)p[order[0]];")], ["test_softmax_and_stats_match_scipy"]),
    "dispatch_weights_uniform": ([("softmax_row(E, scores + (size_t)t * E, p);\n            double tot = 0.0;",
                                   "for (int e = 0; e < E; ++e) p[e] = 1.0 / E;\n            double tot = 0.0;")],
                                 ["test_combine_weight_page_example"]),
    "combine_ignores_weight": ([("double w = (double)cw[(size_t)t * k + r];", "double w = 1.0;")],
                               ["test_combine_rows_weights_and_drops"]),
    "combine_weight_of_rank0": ([("double w = (double)cw[(size_t)t * k + r];", "double w = (double)cw[(size_t)t * k];")],
                                ["test_combine_rows_weights_and_drops"]),
    "slot_token_assumes_k2": ([("int t = idx / k;", "int t = idx / 2;")], ["test_q8_activation_rounding_hand_case"]),
    "q8_row_max_of_first_8": ([("for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));\n"
                                "    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;",
                                "for (int i = 0; i < 8 && i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));\n"
                                "    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;")],
                              ["test_quantize_row_matches_torch"]),
    "nvfp4_row_max_of_first_block": ([("for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));\n"
                                       "    const float s = amax > 0.0f ? amax / 2688.0f : 1.0f;",
                                       "for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));\n"
                                       "    const float s = amax > 0.0f ? amax / 2688.0f : 1.0f;")],
                                     ["test_nvfp4_row_quantisation_is_exact_on_representable_rows"]),
    "nvfp4_block_max_of_half": ([("for (int i = 16 * j; i < 16 * j + 16; ++i) bmax = fmaxf(bmax, fabsf(x[i]));",
                                  "for (int i = 16 * j; i < 16 * j + 8; ++i) bmax = fmaxf(bmax, fabsf(x[i]));")],
                                ["test_nvfp4_row_quantisation_is_exact_on_representable_rows"]),
    "bwd_dwr_of_wr": ([("dwr[(size_t)e * d + i] += dz * x[i];",
                        "dwr[(size_t)e * d + i] += dz * (double)bf16_to_f32(we[i]);")],
                      ["test_backward_matches_torch_autograd"]),
    "bwd_dbias_missing": ([("dbias[e] += dz;", "(void)0;")],
                          ["test_backward_dropped_token_gets_only_the_aux_gradient"]),
    "bwd_cw_not_renormalised": ([("cw[r] = (e >= 0 && S > 0.0) ? p[e] / S : 0.0;",
                                  "cw[r] = (e >= 0 && S > 0.0) ? p[e] : 0.0;")],
                                ["test_backward_matches_torch_autograd"]),
}


def _build_and_run(name, tmpdir):
    edits, _ = MUTANTS[name]
    with open(oracle._SRC) as fh:
        src = fh.read()
    for old, new in edits:
        n = src.count(old)
        if n != 1:
            return None, f"edit of {name!r} matches {n} places"
        src = src.replace(old, new)
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"lib{name}.so")
    with open(c, "w") as fh:
        fh.write(src)
    r = subprocess.run(["gcc", *oracle.CFLAGS, "-I", os.path.dirname(oracle._SRC), "-o", so, c, "-lm"],
                       capture_output=True, text=True)
    if r.returncode:
        return None, r.stderr
    env = dict(os.environ, MOE_ORACLE_LIBRARY=so)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-q", "-p", "no:cacheprovider", "-rf",
                        "-k", "not workload_router_statistics"],
                       capture_output=True, text=True, env=env, cwd=os.path.dirname(HERE), timeout=600)
    if r.returncode not in (0, 1):   # 1: some test failed; anything else: the run itself broke
        return None, f"pin run of {name!r} ended with status {r.returncode}\n{r.stdout[-2000:]}{r.stderr[-1000:]}"
    failed = set(re.findall(r"^FAILED \S*::(test_\w+)", r.stdout, re.M))
    return failed, r.stdout[-3000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    tmpdir = str(tmp_path_factory.mktemp("mutants"))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {n: ex.submit(_build_and_run, n, tmpdir) for n in MUTANTS}
        return {n: f.result() for n, f in futs.items()}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_its_pins(name, mutant_results):
    failed, log = mutant_results[name]
    assert failed is not None, log
    missing = [p for p in MUTANTS[name][1] if p not in failed]
    assert not missing, f"{name}: pins {missing} did not fail\n{log}"


def test_unmutated_copy_passes():
    """The harness itself: the pins pass on an unedited library built the same way."""
    MUTANTS["_unmutated"] = ([], [])
    try:
        import tempfile
        with tempfile.TemporaryDirectory() as d:
            failed, log = _build_and_run("_unmutated", d)
    finally:
        del MUTANTS["_unmutated"]
    assert failed == set(), log
