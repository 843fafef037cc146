"""The oracle's pins catch plausible mistakes: each test plants one mistake in a copy of oracle.c (on the CPU, in a
temporary directory), binds the copy in place of the oracle and checks that at least one of the named pins of
tests/test_oracle_formats.py and tests/test_oracle_router_ffn.py fails on it. The unmodified oracle passes them all
(those files' own runs)."""
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_formats as tf
import tests.test_oracle_router_ffn as tr

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# name: (text in oracle.c, the planted mistake, pins of which at least one must fail)
MUTANTS = {
    "mxfp4_nibble_order": ("return (j % 2 == 0) ? (b >> 4) : (b & 15);",
                           "return (j % 2 == 0) ? (b & 15) : (b >> 4);",
                           [tf.test_mxfp4_element_order_follows_printed_unpack, tf.test_mxfp4_handbuilt_blocks]),
    "e8m0_bias": ("return ldexp(1.0, e - 127);", "return ldexp(1.0, e - 126);",
                  [tf.test_e8m0_rule, tf.test_mxfp4_handbuilt_blocks]),
    "int4_sign": ("return n >= 8 ? n - 16 : n;   /* two's complement */", "return n;",
                  [tf.test_int4_layout_and_decode_closed_form]),
    "q2k_min_sign": ("  return bq - c;\n}", "  return bq + c;\n}",
                     [tf.test_q2k_handbuilt_block, tf.test_q2k_decode_matches_closed_form_random_blocks]),
    "router_ties_to_upper": ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;",
                             [tr.test_router_ties_go_to_lower_index]),
    "router_weights_unnormalised": ("for (int r = 0; r < k; ++r) den += exp(sel[r] - mx);",
                                    "for (int r = 0; r < k; ++r) den = 1.0;",
                                    [tr.test_router_matches_sort_and_scipy_softmax]),
    "silu_as_sigmoid": ("static double silu(double g) { return g / (1.0 + exp(-g)); }",
                        "static double silu(double g) { return 1.0 / (1.0 + exp(-g)); }",
                        [tr.test_ffn_integer_case_is_exact, lambda: tr.test_ffn_random_matches_numpy_path(oracle.MXFP4)]),
    "combine_weight_dropped": ("      y[j] += (double)w[r] * d[j];\n      if (absterm) absterm[j] += fabs((double)w[r]) * da[j];",
                               "      y[j] += d[j];\n      if (absterm) absterm[j] += fabs((double)w[r]) * da[j];",
                               [lambda: tr.test_moe_combine_batch_and_token_agree_with_numpy(oracle.MXFP4)]),
    "e2m1_ties_to_odd": ("if (d < bestd || (d == bestd && (c % 2) == 0)) { bestd = d; best = c; }\n  }\n  if (a > 6.0) best = 7;",
                         "if (d < bestd || (d == bestd && (c % 2) == 1)) { bestd = d; best = c; }\n  }\n  if (a > 6.0) best = 7;",
                         [tf.test_mxfp4_encoder_ties_and_roundtrip, tf.test_mxfp4_encoder_brute_force_small]),
    "mx_scale_one_too_small": ("  int e = k + 127;\n", "  int e = k + 126;\n",
                               [tf.test_mxfp4_encoder_brute_force_small, tf.test_mxfp4_encoder_ties_and_roundtrip]),
    "e4m3_ties_to_odd": ("    double d = fabs(a - orc_e4m3_value(c));\n    if (d < bestd || (d == bestd && (c % 2) == 0))",
                         "    double d = fabs(a - orc_e4m3_value(c));\n    if (d < bestd || (d == bestd && (c % 2) == 1))",
                         [tf.test_e4m3_values_and_quantiser_vs_torch, tf.test_mxfp8_quantiser_ties_go_to_even_codes_vs_torch]),
    "int4_grid_without_1": ("const float grid[6] = {6.0f / 7.0f, 0.9f, 0.95f, 1.0f, 1.05f, 1.1f};",
                            "const float grid[6] = {6.0f / 7.0f, 0.9f, 0.95f, 1.05f, 1.05f, 1.1f};",
                            [tf.test_int4_encoder_is_grid_argmin]),
    "int4_clamp_at_minus_7": ("if (qq < -8.0f) qq = -8.0f;", "if (qq < -7.0f) qq = -7.0f;",
                              [tf.test_int4_encoder_is_grid_argmin]),
    "router_drops_last_term": ("      for (int h = 0; h < H; ++h) {\n        double p = orc_f16_to_f64(wr",
                               "      for (int h = 0; h < H - 1; ++h) {\n        double p = orc_f16_to_f64(wr",
                               [tr.test_router_matches_sort_and_scipy_softmax]),
    "hash_weight": ("w[(int64_t)t * k + r] = (float)(1.0 / k);", "w[(int64_t)t * k + r] = (float)(1.0 / (k + 1));",
                    [tr.test_hash_routing_gathers_table_with_equal_weights]),
    "gate_up_swapped": ("    h[i] = silu(gv[i]) * s;", "    h[i] = silu(s) * gv[i];",
                        [tr.test_ffn_integer_case_is_exact, lambda: tr.test_ffn_random_matches_numpy_path(oracle.MXFP4)]),
    "down_transposed": ("      double p = D[(int64_t)j * I + i] * h[i];", "      double p = D[(int64_t)i * H + j % H] * h[i];",
                        [lambda: tr.test_ffn_random_matches_numpy_path(oracle.MXFP4)]),
    "prefill_h_unquantised": ("        double p = weight_at(1, down[r], I, j, i) * hq[i];",
                              "        double p = weight_at(1, down[r], I, j, i) * h[i];",
                              [tr.test_prefill_token_matches_torch_float8_path]),
    "prefill_x_unquantised": ("    orc_expert_ffn(1, H, I, gate[r], up[r], down[r], xq, NULL, NULL, h, NULL, NULL);",
                              "    orc_expert_ffn(1, H, I, gate[r], up[r], down[r], x, NULL, NULL, h, NULL, NULL);",
                              [tr.test_prefill_token_matches_torch_float8_path]),
    "q2k_codes_floored": ("        float qq = rne_int(t / step);\n        if (qq < 0.0f) qq = 0.0f;\n        if (qq > 3.0f) qq = 3.0f;",
                          "        float qq = floorf(t / step);\n        if (qq < 0.0f) qq = 0.0f;\n        if (qq > 3.0f) qq = 3.0f;",
                          [tf.test_q2k_size_and_encoder_bounds]),
    "q2k_offset_dropped": ("        float t = x[i] + off;", "        float t = x[i];",
                           [tf.test_q2k_size_and_encoder_bounds]),
    "q8_0_scale_over_128": ("orc_f32_to_f16_rne(amax / 127.0f);", "orc_f32_to_f16_rne(amax / 128.0f);",
                            [tf.test_q8_0_encoder_against_torch, tf.test_q8_0_encoder_ties_go_to_even_and_clamp]),
    "q8_0_codes_unsigned": ("return (int)(int8_t)blk[2 + j];", "return (int)blk[2 + j];",
                            [tf.test_q8_0_layout_and_decode_closed_form]),
    "q8_0_codes_truncated": ("        qq = rne_int(x[j] / d);", "        qq = truncf(x[j] / d);",
                             [tf.test_q8_0_encoder_against_torch, tf.test_q8_0_encoder_ties_go_to_even_and_clamp]),
}


def _bind_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name  # every occurrence gets the mistake (the combine appears in two functions)
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(old, new))
    so = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    str(path), "-o", str(so), "-lm"], check=True)
    return oracle.bind(str(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(tmp_path, monkeypatch, name):
    old, new, pins = MUTANTS[name]
    oracle.lib()  # the real oracle is built and bound first; the mutant replaces it for this test only
    monkeypatch.setattr(oracle, "_lib", _bind_mutant(tmp_path, name, old, new))
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the planted mistake %s" % name
