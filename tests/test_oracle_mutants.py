"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle source (never in the
oracle itself), builds it, and runs the CPU pins of test_oracle_pins.py
against it: at least one pin must fail.  A mistake no pin notices would mean
the oracle is not pinned where it matters."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.cpp")

MUTANTS = {
    "tie_break_to_higher_index": ("return a < b;   // equal logits", "return a > b;   // equal logits"),
    "softmax_over_all_experts": ("for (int j = 0; j < k; ++j) z += std::exp",
                                 "for (int j = 0; j < E; ++j) z += std::exp"),
    "gate_and_up_swapped": ("h_row[n] = double_to_bf16(silu(g) * u);", "h_row[n] = double_to_bf16(silu(u) * g);"),
    "relu_dropped": ("const double r = a > 0.0 ? a : 0.0;", "const double r = a;"),
    "down_weights_transposed": ("s += bf16_to_double(h_row[n]) * bf16_to_double(wrow[n]);",
                                "s += bf16_to_double(h_row[n]) * bf16_to_double(w2_e[(size_t)n * H + c]);"),
    "shared_term_dropped": ("if (y_shared_t) s += bf16_to_double(y_shared_t[c]);", "if (y_shared_t) s += 0.0;"),
    "bucket_order_reversed": ("const int32_t d = offsets[e] + fill[e];",
                              "const int32_t d = offsets[e + 1] - 1 - fill[e];"),
    "bf16_truncates": ("if (frac > 0.5 || (frac == 0.5 && std::fmod(qi, 2.0) != 0.0)) qi += 1.0;",
                       "if (false) qi += 1.0;"),
    "capacity_off_by_one": ("if (counts[e] > capacity)", "if (counts[e] >= capacity)"),
    "duplicates_not_detected": ("if (ids[(size_t)t * k + jj] == e) ok = false;", "if (false) ok = false;"),
    "weights_paired_with_wrong_slot": ("s += (double)w_t[j] * bf16_to_double", "s += (double)w_t[k - 1 - j] * bf16_to_double"),
    "sigmoid_bias_ignored": ("key[e] = score[e] + (bias ? bias[e] : 0.0f);", "key[e] = score[e];"),
    "sigmoid_weights_from_biased_key": ("(double)route_scale * (double)score[order[j]] / z",
                                        "(double)route_scale * (double)key[order[j]] / z"),
    "gate_transposed": ("bf16_to_double(wg[(size_t)e * H + h])", "bf16_to_double(wg[(size_t)h * E + e])"),
    "residual_dropped": ("if (residual_t) s += bf16_to_double(residual_t[c]);", "if (residual_t) s += 0.0;"),
    "fp8_gate_and_up_swapped": ("h_row[n] = double_to_bf16(silu(gate) * upv);",
                                "h_row[n] = double_to_bf16(silu(upv) * gate);"),
    "fp8_exponent_bias_8": ("std::ldexp(1.0 + m / 8.0, e - 7)", "std::ldexp(1.0 + m / 8.0, e - 8)"),
    "fp8_subnormals_read_as_normals": ("(e == 0) ? std::ldexp((double)m, -9)", "(e == 0) ? std::ldexp(1.0 + m / 8.0, -7)"),
    "fp8_nan_code_finite": ("if (e == 15 && m == 7) return std::nan(\"\");", "if (false) return std::nan(\"\");"),
    "fp8_up_scale_from_first_row": ("return acc * (double)s13_e[wr];", "return acc * (double)s13_e[0];"),
    "fp8_down_scale_from_first_row": ("double_to_bf16(acc * (double)s2_e[c])", "double_to_bf16(acc * (double)s2_e[0])"),
    "fp4_nibbles_swapped": ("const uint8_t code = (c & 1) ? (b >> 4) : (b & 15);",
                            "const uint8_t code = (c & 1) ? (b & 15) : (b >> 4);"),
    "fp4_exponent_bias_0": ("std::ldexp(1.0 + 0.5 * m, e - 1)", "std::ldexp(1.0 + 0.5 * m, e)"),
    "fp4_subnormal_read_as_normal": ("(e == 0) ? 0.5 * m :", "(e == 0) ? std::ldexp(1.0 + 0.5 * m, -1) :"),
    "nvfp4_block_of_8": ("fp8_e4m3_to_double(bscale_row[c >> 4])", "fp8_e4m3_to_double(bscale_row[c >> 3])"),
    "nvfp4_unpadded_scale_rows": ("return 16 * (size_t)((K + 255) / 256);", "return (size_t)(K / 16);"),
    "nvfp4_up_row_scale_dropped": ("return acc * (double)s13[row];", "return acc;"),
    "nvfp4_down_row_scale_from_first_row": ("double_to_bf16(acc * (double)s2[row])",
                                            "double_to_bf16(acc * (double)s2[(size_t)e * H])"),
    "first_slot_dropped_in_combine": ("for (int j = 0; j < k; ++j) {\n            if (dest_t[j] < 0) continue;",
                                      "for (int j = 1; j < k; ++j) {\n            if (dest_t[j] < 0) continue;"),
}

PINS = [
    (P.test_bf16_rounding_matches_torch_on_float_values, {}),
    (P.test_bf16_rounding_single_rounding_from_double, {}),
    (P.test_route_bruteforce_with_ties, dict(E=16, k=2)),
    (P.test_route_bruteforce_with_ties, dict(E=33, k=5)),
    (P.test_route_negative_zero_ties_positive_zero, {}),
    (P.test_route_closed_form_two_experts, {}),
    (P.test_route_decode_closed_form_golden, {}),
    (P.test_dispatch_bruteforce_and_invariants, dict(T=64, E=16, k=2)),
    (P.test_dispatch_capacity_exceeded_moves_no_payload, {}),
    (P.test_dispatch_invalid_routes, dict(kind="duplicate")),
    (P.test_dispatch_invalid_routes, dict(kind="negative")),
    (P.test_ffn_single_expert_is_dense_mlp, dict(act=0)),
    (P.test_ffn_single_expert_is_dense_mlp, dict(act=1)),
    (P.test_ffn_identical_experts_give_dense_mlp_for_any_routing, {}),
    (P.test_layer_relu2_analytic_exact, dict(k=2)),
    (P.test_shared_experts_sum_before_rounding, {}),
    (P.test_combine_identity_experts_return_x, dict(k=4)),
    (P.test_combine_weights_are_applied_per_slot, {}),
    (P.test_combine_residual_is_added_once, {}),
    (P.test_layer_internal_routing_equals_preselected, {}),
    (P.test_route_sigmoid_without_bias_selects_like_softmax, {}),
    (P.test_route_sigmoid_dominant_bias_selects_its_set_and_weights_ignore_it, {}),
    (P.test_route_sigmoid_negative_bias_excludes_the_top_experts, {}),
    (P.test_route_sigmoid_closed_form_weights, {}),
    (P.test_gate_projection_matches_float64_matmul, {}),
    (P.test_fp8_decode_closed_forms, {}),
    (P.test_fp8_decode_matches_torch, {}),
    (P.test_fp8_ffn_equals_bf16_path_on_exact_weights, dict(act=0)),
    (P.test_fp8_ffn_equals_bf16_path_on_exact_weights, dict(act=1)),
    (P.test_fp8_layer_equals_bf16_layer_on_exact_weights, {}),
    (P.test_fp4_decode_values, {}),
    (P.test_nvfp4_ffn_equals_bf16_path_on_exact_weights, dict(act=0, H=48, I=64)),
    (P.test_nvfp4_ffn_equals_bf16_path_on_exact_weights, dict(act=1, H=288, I=32)),
    (P.test_nvfp4_layer_equals_bf16_layer_on_exact_weights, {}),
    (P.test_nvfp4_layer_preselected_routes_and_capacity, {}),
]


def run_pins(mod):
    failed = []
    for fn, kw in PINS:
        try:
            fn(mod, **kw)
        except AssertionError:
            failed.append(fn.__name__)
    return failed


def test_unmutated_oracle_passes_every_pin(oracle_mod):
    assert run_pins(oracle_mod) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation point of {name} not found once"
    msrc = tmp_path / "mutant.cpp"
    msrc.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-fPIC", "-shared", "-o", str(lib), str(msrc)])
    mod = oracle.variant(str(lib), str(msrc))
    failed = run_pins(mod)
    assert failed, f"planted mistake '{name}' passed every pin"
