"""Plant plausible mistakes in a COPY of the oracle (compiled on the CPU) and check that
the pins in test_oracle_pins.py catch each one."""
import pytest

import oracle
import sys, os
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import test_oracle_pins as pins

MUTATIONS = {
    "tie_to_smaller_index": [("if (a->idx > b->idx) return -1;\n  if (a->idx < b->idx) return 1;",
                              "if (a->idx < b->idx) return -1;\n  if (a->idx > b->idx) return 1;")],
    "own_block_not_kept": [("out[take] = (int32_t)bt;", "out[take] = (int32_t)(take < bt ? c[take].idx : bt);")],
    "causal_strict": [("if (j <= t) J[nJ++] = j;", "if (j < t || j == 0) J[nJ++] = j;")],
    "scale_dropped": [("s[i] = d->scale * acc;", "s[i] = acc;")],
    "gate_sign": [("* sigmoid(gt);", "* sigmoid(-gt);")],
    "mean_over_B_not_present": [("sum / (double)n", "sum / (double)B")],
    "values_from_keys": [("const uint16_t* vr = V + (g * ctx_cap + off + J[i]) * D;",
                          "const uint16_t* vr = K + (g * ctx_cap + off + J[i]) * D;")],
    "double_rounding": [("double r = nearbyint(x / quantum) * quantum;",
                         "double r = nearbyint((double)(float)x / quantum) * quantum;")],
    "keeps_one_block_too_few": [("int64_t take = bt < d->k - 1 ? bt : d->k - 1;",
                                 "int64_t take = bt < d->k - 2 ? bt : (d->k > 2 ? d->k - 2 : 0);")],
    "softmax_no_max_shift_wrong_lse": [("if (lse) lse[r * Hg + h] = m + log(l);", "if (lse) lse[r * Hg + h] = log(l);")],
    "e4m3_exponent_bias": [("ldexp(1.0 + M / 8.0, E - 7)", "ldexp(1.0 + M / 8.0, E - 8)")],
    "e4m3_round_down": [("double r = nearbyint(a / quantum) * quantum;", "double r = floor(a / quantum) * quantum;")],
    "e4m3_no_subnormal_floor": [("if (lead < -6) lead = -6;", "if (lead < -9) lead = -9;")],
    "e4m3_no_saturation": [("if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 480.0;")],
}

PIN_CALLS = [
    lambda: pins.test_bf16_rounding_is_a_single_rounding(),
    lambda: pins.test_block_index_integer_proxies_exact(8),
    lambda: pins.test_block_index_partial_range_only_touches_its_blocks(),
    lambda: pins.test_score_invariant_block_mean_equals_token_scores_over_B(),
    lambda: pins.test_selection_matches_full_sort(7, -4, 4),
    lambda: pins.test_selection_closed_forms(),
    lambda: pins.test_attention_full_selection_equals_dense_causal(),
    lambda: pins.test_attention_two_token_worked_example(),
    lambda: pins.test_attention_sparse_selection_is_a_subset_softmax(),
    lambda: pins.test_coverage_closed_forms(),
    lambda: pins.test_e4m3_decoding_matches_torch(),
    lambda: pins.test_e4m3_rounding_matches_torch_on_float32_values(),
    lambda: pins.test_e4m3_saturation_and_special_values(),
    lambda: pins.test_e4m3_cache_of_integer_proxy_means(),
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    caught = []
    with oracle.mutated(MUTATIONS[name], tmp_path):
        for i, call in enumerate(PIN_CALLS):
            try:
                call()
            except (AssertionError, ValueError):
                caught.append(i)
    assert caught, f"no pin caught mutation {name}"


def test_unmutated_oracle_passes_every_pin():
    for call in PIN_CALLS:
        call()
