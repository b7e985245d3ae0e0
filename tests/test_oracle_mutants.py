"""The pins must reject a broken oracle.

Each case edits one plausible slip into a copy of the oracle source, compiles
it on the CPU, swaps it in, and checks that at least one pin of
``test_oracle_pins`` fails.  The real oracle is never modified.
"""
import pytest

from oracle import oracle as orc
from tests import test_oracle_bwd_pins as bwd_pins
from tests import test_oracle_mixed_pins as mixed_pins
from tests import test_oracle_pins as pins

MUTANTS = {
    "reversed tap order": ("load_value(weight, c * ws[0] + k * ws[1], wdtype)",
                           "load_value(weight, c * ws[0] + (K - 1 - k) * ws[1], wdtype)"),
    "source index off by one": ("int64_t j = t - (K - 1) + k;", "int64_t j = t - K + k;"),
    "bias dropped": ("double z = bias ? load_value(bias, c * bias_stride, wdtype) : 0.0;",
                     "double z = 0.0;"),
    "initial_states read newest first": (
        "if (init) return load_value(init, b * is[0] + c * is[1] + (K - 1 + j) * is[2], dtype);",
        "if (init) return load_value(init, b * is[0] + c * is[1] + (-1 - j) * is[2], dtype);"),
    "seq_idx compared one step late": (
        "if (seq_idx[b * ss[0] + j * ss[1]] != sid_t) continue;",
        "if (seq_idx[b * ss[0] + (j + 1 < t ? j + 1 : t) * ss[1]] != sid_t) continue;"),
    "silu sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "double rounding through float": ("double a = fabs(v);", "double a = fabs((double)(float)v);"),
    "ties away from zero": ("double n = nearbyint(ldexp(a, -q));", "double n = round(ldexp(a, -q));"),
    "no gradual underflow": ("if (E < f.emin) E = f.emin;", "if (E < f.emin - 100) E = f.emin;"),
    "final_states off by one": ("int64_t src = L - (K - 1) + j;", "int64_t src = L - K + j;"),
    "final_states from history only when short": (
        "else if (init)\n            bits = load_bits(init,", "else if (0)\n            bits = load_bits(init,"),
    "last tap skipped": ("for (int k = 0; k < K; ++k) {", "for (int k = 0; k < K - 1; ++k) {"),
    # backward pass
    "silu gradient without the z term": ("return s + z * s * (1.0 - s);", "return s;"),
    "dz ignores the activation": ("const double dz = silu_act ? g * silu_grad(z) : g;", "const double dz = g;"),
    "dx through the reversed kernel": ("dh[j + H] += wc[tap] * dz;", "dh[j + H] += wc[K - 1 - tap] * dz;"),
    "dweight paired with the next input": (
        "if (dweight) dweight[c * K + tap] += dz * h;",
        "if (dweight) dweight[c * K + tap] += dz * history_value(x, xs, init, is, b, c, j + (j + 1 < L), K, dtype);"),
    "dbias from dout instead of dz": ("db += dz;", "db += g;"),
    "dfinal one step late": ("const int64_t src = L - H + j; /* final_states[j] is h[src] */",
                             "const int64_t src = L - H + j + 1;"),
    "dinitial_states newest first": ("if (dinit) dinit[(b * C + c) * H + i] = dh[i];",
                                     "if (dinit) dinit[(b * C + c) * H + i] = dh[H - 1 - i];"),
    "backward ignores seq_idx": ("if (!seq_idx) return 1;", "return 1;"),
    # separate weight dtype
    "weight decoded in the input dtype": ("double w = load_value(weight, c * ws[0] + k * ws[1], wdtype);",
                                          "double w = load_value(weight, c * ws[0] + k * ws[1], dtype);"),
    "backward bias decoded in the input dtype": (
        "const double bc = bias ? load_value(bias, c * bias_stride, wdtype) : 0.0;",
        "const double bc = bias ? load_value(bias, c * bias_stride, dtype) : 0.0;"),
}

# pin bodies run against each mutant (any failing one is enough)
CHECKS = [
    (pins.test_golden_hand_worked_example, {}),
    (pins.test_impulse_reproduces_reversed_kernel, {"dt": "f32", "K": 4}),
    (pins.test_identity_kernel_is_bit_exact, {"dt": "bf16", "layout": "channel"}),
    (pins.test_zero_input_gives_activated_bias, {"dt": "f32"}),
    (pins.test_matches_numpy_convolve_and_toeplitz, {"K": 3}),
    (pins.test_two_chunks_equal_one_pass, {"dt": "bf16", "K": 4}),
    (pins.test_final_states_closed_form, {"dt": "f16"}),
    (pins.test_packed_segments_equal_separate_runs, {"dt": "f32"}),
    (pins.test_seq_idx_degenerate_cases, {"dt": "f16"}),
    (pins.test_silu_special_values_and_library, {}),
    (pins.test_round_bf16_bruteforce_and_ties, {}),
    (pins.test_round_f16_matches_numpy_direct_conversion, {}),
    (bwd_pins.test_bwd_matches_framework_autograd, {"dt": "f32", "K": 4, "act": "silu", "layout": "time"}),
    (bwd_pins.test_linear_bwd_is_transposed_band_matrix, {"K": 3, "with_seq": True}),
    (bwd_pins.test_bwd_matches_central_differences, {"K": 3, "act": "silu", "L": 9}),
    (bwd_pins.test_bwd_of_chunks_chained_by_states_equals_one_pass, {"dt": "bf16", "K": 4}),
    (bwd_pins.test_dfinal_alone_lands_on_the_copied_inputs, {"dt": "f32"}),
    (bwd_pins.test_packed_segments_bwd_equal_separate_runs, {"dt": "f16"}),
    (mixed_pins.test_mixed_forward_matches_framework_conv1d, {"dt": "bf16", "wdt": "f32"}),
    (mixed_pins.test_mixed_backward_matches_framework_autograd, {"dt": "f32", "wdt": "f16"}),
    (mixed_pins.test_weights_exact_in_both_formats_give_the_one_dtype_result, {"dt": "f16", "wdt": "bf16"}),
    (mixed_pins.test_weights_exact_in_both_formats_give_the_one_dtype_gradients, {"dt": "bf16", "wdt": "f16"}),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = orc.source_text()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    lib = orc.compile_variant(src.replace(old, new), str(tmp_path), "mutant")
    failed = []
    with orc.swapped_library(lib):
        for fn, kw in CHECKS:
            try:
                fn(**kw)
            except (AssertionError, orc.OracleError):
                failed.append(fn.__name__)
    assert failed, f"no pin caught the mutant '{name}'"
