"""Plant plausible mistakes in a copy of the oracle and check that a pin catches each.

Every mutation below is a one-token slip of the kind a restatement of the pages could
contain (a flipped sign, a swapped operand, an off-by-one row, a dropped term, a wrong tie
rule).  The copy is compiled on the CPU into a temporary shared object; the real oracle is
never modified.
"""
import functools

import pytest

import oracle
import oracle_pins as pins

chi2_quick = functools.partial(pins.pin_chi2_sampler, trials=200_000)
chi2_quick.__name__ = "pin_chi2_sampler_quick"
tree_chi2_quick = functools.partial(pins.pin_tree_sample_chi2, trials=100_000)
tree_chi2_quick.__name__ = "pin_tree_sample_chi2_quick"

MUTATIONS = [
    ("residual_sign", "double d = p[j] - q[j];\n            r[j] = d > 0.0 ? d : 0.0;",
     "double d = q[j] - p[j];\n            r[j] = d > 0.0 ? d : 0.0;",
     [pins.pin_bruteforce_lossless, chi2_quick]),
    ("accept_test_swapped", "if (u * qx < px)", "if (u * px < qx)",
     [chi2_quick, pins.pin_one_hot_equals_greedy]),
    ("accept_prob_inverted", "return px / qx < 1.0 ? px / qx : 1.0;",
     "return qx / px < 1.0 ? qx / px : 1.0;", [pins.pin_bruteforce_lossless, pins.pin_worked_example]),
    ("temperature_dropped_in_sum", "S += exp(l[j] / T - m);", "S += exp(l[j] - m);",
     [pins.pin_row_stats, pins.pin_bruteforce_lossless]),
    ("bonus_from_wrong_row", "softmax_row(t_logits + (size_t)gamma * V, V, T, p, NULL, NULL)",
     "softmax_row(t_logits + (size_t)(gamma - 1) * V, V, T, p, NULL, NULL)",
     [pins.pin_bruteforce_lossless]),
    ("stop_row_off_by_one", "int k = gamma, residual = 0;", "int k = gamma - 1, residual = 0;",
     [pins.pin_identical_rows_accept_all, pins.pin_round_invariants]),
    ("cdf_returns_next", "*margin = fmin(fabs(target - prev), fabs(C - target)) / R;\n            return j;",
     "*margin = 1.0;\n            return j + 1 < V ? j + 1 : j;", [chi2_quick]),
    ("uniform_half_range", "return (double)(w[0] >> 8) * (1.0 / 16777216.0);",
     "return (double)(w[0] >> 9) * (1.0 / 16777216.0);", [pins.pin_uniform_definition, chi2_quick]),
    ("philox_key_not_bumped", "k0 += W0;", "k0 += 0u;", [pins.pin_philox_kat]),
    ("philox_words_swapped", "uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi0 ^ c1 ^ k0;",
     [pins.pin_philox_kat]),
    ("greedy_stop_token", "out[n] = a[n];\n        accepted_len[b] = n;",
     "out[n] = a[n > 0 ? n - 1 : 0];\n        accepted_len[b] = n;", [pins.pin_greedy_textbook]),
    ("argmax_ties_to_highest", "if (l[j] > l[best])", "if (l[j] >= l[best])",
     [pins.pin_greedy_textbook]),
    ("tree_compares_own_argmax", "node_tokens[(int64_t)b * N + v] == a[parent[v]];",
     "node_tokens[(int64_t)b * N + v] == a[v];", [pins.pin_tree_bruteforce, pins.pin_tree_printed_depths]),
    ("tree_depth_tie_to_highest", "if (acc[v] && depth[v] > depth[best])",
     "if (acc[v] && depth[v] >= depth[best])", [pins.pin_tree_bruteforce]),
    ("tree_parent_not_required", "acc[v] = acc[parent[v]] && ", "acc[v] = ",
     [pins.pin_tree_bruteforce]),
    ("lse_missing_temperature", "if (l[j] / T > m)\n            m = l[j] / T;",
     "if (l[j] > m)\n            m = l[j];", [pins.pin_row_stats]),
    ("tree_siblings_against_original_p", "            p[j] = r[j] / R;", "            p[j] = p[j];",
     [pins.pin_tree_sample_lossless, tree_chi2_quick]),
    ("tree_q_not_renormalised", "q[j] = Q > 0.0 ? q[j] / Q : 0.0;", "q[j] = Q > 0.0 ? q[j] : 0.0;",
     [pins.pin_tree_sample_lossless]),
    ("tree_rejected_token_kept_in_q", "        q[x] = 0.0;", "        q[x] = q[x];",
     [pins.pin_tree_sample_lossless]),
    ("tree_uniform_index", "(uint32_t)(c - 1), 0u);", "(uint32_t)c, 0u);",
     [pins.pin_chain_tree_sample_equals_chain]),
    ("tree_sampler_accept_swapped", "if (u * q[x] < p[x]) {", "if (u * p[x] < q[x]) {",
     [tree_chi2_quick, pins.pin_chain_tree_sample_equals_chain]),
    ("ngram_earliest_match", "for (int i = L - n - 1; i >= 0 && match < 0; --i) {",
     "for (int i = 0; i <= L - n - 1 && match < 0; ++i) {",
     [pins.pin_ngram_worked_examples, pins.pin_ngram_bruteforce]),
    ("ngram_tail_matches_itself", "for (int i = L - n - 1; i >= 0 && match < 0; --i) {",
     "for (int i = L - n; i >= 0 && match < 0; --i) {",
     [pins.pin_ngram_worked_examples, pins.pin_ngram_bruteforce]),
    ("ngram_no_fallback", "        if (pad && L >= 1)\n            for (; c < k; ++c)",
     "        if (0 && pad && L >= 1)\n            for (; c < k; ++c)",
     [pins.pin_ngram_worked_examples, pins.pin_ngram_bruteforce]),
    ("typical_entropy_in_bits", "H -= p[j] * log(p[j]);", "H -= p[j] * log2(p[j]);",
     [pins.pin_typical_entropy, pins.pin_typical_threshold_closed_forms]),
    ("typical_entropy_sign", "double tau = delta * exp(-H);", "double tau = delta * exp(H);",
     [pins.pin_typical_threshold_closed_forms]),
    ("typical_threshold_max", "if (epsilon < tau)\n                tau = epsilon;",
     "if (epsilon > tau)\n                tau = epsilon;", [pins.pin_typical_threshold_closed_forms]),
    ("typical_accept_on_equality", "if (!(px > tau)) {", "if (!(px >= tau)) {",
     [pins.pin_typical_threshold_closed_forms]),
    ("typical_stop_off_by_one", "                k = i;\n                break;",
     "                k = i + 1 > gamma ? gamma : i + 1;\n                break;",
     [pins.pin_typical_zero_threshold, pins.pin_typical_draw_law]),
]


@pytest.mark.parametrize("name,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, catchers):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    bad = oracle.variant(src.replace(old, new), str(tmp_path))
    failures = []
    for pin in catchers:
        try:
            pin(bad)
        except AssertionError as e:  # the pin caught the planted mistake
            failures.append((pin.__name__, str(e)[:80]))
    assert failures, f"no pin caught the planted mistake {name}"
