"""Planted mistakes: each plausible slip in the oracle must fail some pin.

Every case below edits one spot of a copy of oracle.c (on the CPU, in a temp
directory), builds it, points the oracle module at the copy, and runs the pins
of test_oracle_pins.py.  The test passes only if at least one pin fails on the
mutant, which shows the pins constrain that part of the oracle.
"""
import pytest

import oracle
import test_oracle_pins as pins

PINS = [
    pins.test_logits_exact_on_integers,
    pins.test_logits_hand_worked_order,
    pins.test_logits_error_bound_vs_fp64,
    lambda: pins.test_topk_matches_brute_force_with_ties(13, 4),
    pins.test_topk_signed_zero_tie,
    pins.test_topk_weights_k1_is_one,
    pins.test_topk_weights_are_softmax_of_chosen,
    pins.test_topk_closed_form_two_experts,
    lambda: pins.test_dispatch_brute_force(33, 9, 3),
    pins.test_dispatch_invariants,
    pins.test_layer_single_expert_is_dense_swiglu,
    pins.test_layer_identical_experts_is_dense,
    pins.test_layer_k_equals_E_is_full_mixture,
    pins.test_layer_power_of_two_scaling_is_exact,
    pins.test_expert_linear_matches_torch_matmul,
    pins.test_expert_linear_permutation_and_scale_experts,
    pins.test_dispatch_gemm_composes_route_dispatch_linear,
]

MUTANTS = {
    "gate_up_swapped": ("double silu = g / (1.0 + exp(-g));\n        h[n] = silu * u;",
                        "double silu = u / (1.0 + exp(-u));\n        h[n] = silu * g;"),
    "silu_sign": ("g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    "tie_goes_to_higher_id": ("l[e] > l[best]) best = e;", "l[e] >= l[best]) best = e;"),
    "contiguous_lane_chunks": ("for (int i = j; i < d; i += 32)\n",
                               "for (int i = j * (d / 32); i < (j + 1) * (d / 32); ++i)\n"),
    "multiply_then_add": ("acc = fmaf(bf16_bits_to_float(xrow[i]), wrow[i], acc);",
                          "acc = bf16_bits_to_float(xrow[i]) * wrow[i] + acc;"),
    "bias_dropped": ("if (bias) l = l + bias[e];", "(void)bias;"),
    "first_chunk_dropped": ("for (int i = j; i < d; i += 32)\n", "for (int i = j + 32; i < d; i += 32)\n"),
    "w2_transposed": ("acc += (double)bf16_bits_to_float(r2[n]) * h[n];",
                      "acc += (double)bf16_bits_to_float(w2e[(int64_t)n * d + c]) * h[n];"),
    "weights_not_renormalised": ("w[j] = exp((double)l[ids[j]] - top) / z;", "w[j] = exp((double)l[ids[j]] - top);"),
    "rows_descending_in_expert": ("int32_t r = offsets[e] + fill[e];", "int32_t r = offsets[e + 1] - 1 - fill[e];"),
    "combine_uses_first_weight": ("yrow[c] += w[j] * out[c];", "yrow[c] += w[0] * out[c];"),
    "w3_uses_w1_row": ("const uint16_t* r3 = w3e + (int64_t)n * d;", "const uint16_t* r3 = w1e + (int64_t)n * d;"),
    "linear_weight_transposed": ("const uint16_t* wrow = we + (int64_t)c * d;\n            double acc = 0.0;\n"
                                 "            for (int i = 0; i < d; ++i) acc += (double)bf16_bits_to_float(wrow[i])",
                                 "const uint16_t* wrow = we + c;\n            double acc = 0.0;\n"
                                 "            for (int i = 0; i < d; ++i) acc += (double)bf16_bits_to_float(wrow[(int64_t)i * n])"),
    "linear_expert_stride_d": ("const uint16_t* we = w + (int64_t)expert[p] * n * d;",
                               "const uint16_t* we = w + (int64_t)expert[p] * d;"),
    "linear_last_term_dropped": ("for (int i = 0; i < d; ++i) acc += (double)bf16_bits_to_float(wrow[i])",
                                 "for (int i = 0; i < d - 1; ++i) acc += (double)bf16_bits_to_float(wrow[i])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    lib = str(tmp_path / f"liboracle_{name}.so")
    oracle.compile_variant(src.replace(old, new), lib)
    prev = oracle.use_library(lib)
    failures = []
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError as exc:  # the pin caught the mutant
                failures.append(getattr(pin, "__name__", "pin") + ": " + str(exc)[:80])
    finally:
        oracle.restore_library(prev)
    assert failures, f"no pin catches the planted mistake {name!r}"
