"""Plant plausible mistakes in copies of the oracle source and check that the
pins in test_oracle_pins.py catch every one of them.

Each mutant is a one-line change of ``oracle/spec_oracle.c`` (a dropped term,
a wrong sign or index, a transposed operand, a flipped tie-break), compiled
into a temporary library on the CPU.  The committed oracle itself is never
modified.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_oracle.c")

MUTANTS = {
    "residual_sign": ("        double d = pt[(size_t)n * V + j] - pd[(size_t)n * V + j];",
                      "        double d = pd[(size_t)n * V + j] - pt[(size_t)n * V + j];"),
    "accept_transposed": ("if (!(u * q < p)) { n = i; break; }",
                          "if (!(u * p < q)) { n = i; break; }"),
    "accept_non_strict": ("if (!(u * q < p)) { n = i; break; }",
                          "if (!(u * q <= p)) { n = i; break; }"),
    "residual_wrong_row": ("        double d = pt[(size_t)n * V + j] - pd[(size_t)n * V + j];",
                           "        double d = pt[(size_t)(n + 1) * V + j] - pd[(size_t)n * V + j];"),
    "bonus_wrong_row": ("tok = inverse_cdf(pt + (size_t)k * V,",
                        "tok = inverse_cdf(pt + (size_t)(k > 0 ? k - 1 : 0) * V,"),
    "temperature_dropped": ("out[j] = exp(logit_at(base, dtype, off + (size_t)j) / T - m);",
                            "out[j] = exp(logit_at(base, dtype, off + (size_t)j) - m / T);"),
    "cdf_unnormalised_u": ("double t = u * R;", "double t = u;"),
    "argmax_last_tie": ("if (z > bv) { bv = z; best = j; }", "if (z >= bv) { bv = z; best = j; }"),
    "tree_last_tie": ("if (ok[v] && depth[v] > depth[best]) best = v;",
                      "if (ok[v] && depth[v] >= depth[best]) best = v;"),
    "tree_ignores_ancestors": ("ok[v] = ok[p] && (tok[v] == g[p]);", "ok[v] = (tok[v] == g[p]);"),
    "tree_bonus_from_parent": ("out_tokens[(size_t)b * W + d] = g[best];",
                               "out_tokens[(size_t)b * W + d] = g[best > 0 ? par[best] : 0];"),
    "greedy_emits_draft": ("else if (i == n) v = g[n];",
                           "else if (i == n) v = (n < k) ? tokens[(size_t)b * k + n] : g[n];"),
    "expected_tokens_short": ("for (int i = 0; i <= gamma; ++i) {", "for (int i = 0; i < gamma; ++i) {"),
    "mask_no_self": ("      int cur = v, d = 0;\n      row[cur / 32] |= 1u << (cur % 32);\n",
                     "      int cur = v, d = 0;\n"),
    "mask_parent_only": ("        ++d;\n      }", "        ++d;\n        break;\n      }"),
    "kv_no_offset": ("const long long src = (long long)(base + path[i] - 1) * entry_bytes;",
                     "const long long src = (long long)(base + path[i]) * entry_bytes;"),
    "kv_scatter": ("memcpy(cache_out + row + dst, cache_in + row + src, (size_t)entry_bytes);",
                   "memcpy(cache_out + row + src, cache_in + row + dst, (size_t)entry_bytes);"),
    "kv_len_counts_bonus": ("new_len[b] = base + d;\n", "new_len[b] = base + d + 1;\n"),
    "kv_previous_node": ("const long long src = (long long)(base + path[i] - 1) * entry_bytes;",
                         "const long long src = (long long)(base + path[i - 1]) * entry_bytes;"),
    "lm_head_transposed": ("z += logit_at(w_lm, OR_BF16, (size_t)j * d + c) * h[c];",
                           "z += logit_at(w_lm, OR_BF16, (size_t)c * V + j) * h[c];"),
    "lm_head_last_tie": ("if (z > best) { second = best; best = z; bj = j; }",
                         "if (z >= best) { second = best; best = z; bj = j; }"),
    "lm_head_emits_draft": ("else if (i == na) v = argmax[(size_t)b * rows + na];",
                            "else if (i == na) v = na < k ? tokens[(size_t)b * k + na] : argmax[(size_t)b * rows + na];"),
    "grow_value_not_cumulative": ("val[n] = val[front[j]] + log(q[best]);", "val[n] = log(q[best]);"),
    "grow_frontier_by_creation": ("if (cand_before(val[order[c]], order[c], val[order[a]], order[a])) {\n              int t = order[a]; order[a] = order[c]; order[c] = t;\n            }\n        nfront",
                                  "if (0) {\n              int t = order[a]; order[a] = order[c]; order[c] = t;\n            }\n        nfront"),
    "grow_token_highest_tie": ("if (!used[x] && (best < 0 || q[x] > q[best])) best = x;",
                               "if (!used[x] && (best < 0 || q[x] >= q[best])) best = x;"),
    "grow_wrong_depth": ("par[n] = front[j]; tok[n] = best; dep[n] = l + 1;",
                         "par[n] = front[j]; tok[n] = best; dep[n] = l;"),
    "grow_keep_by_creation": ("          int t = order[a]; order[a] = order[c]; order[c] = t;\n        }\n    if (nn > M && M > 0)",
                              "          (void)0;\n        }\n    if (nn > M && M > 0)"),
    "pq_first_row_only": ("    for (int i = 0; i < k; ++i) {\n      int32_t x = tokens[(size_t)b * k + i];\n      double p = pt[(size_t)i * V + x];\n      double q = pd[(size_t)i * V + x];\n      if (p_out)",
                          "    for (int i = 0; i < k && i < 1; ++i) {\n      int32_t x = tokens[(size_t)b * k + i];\n      double p = pt[(size_t)i * V + x];\n      double q = pd[(size_t)i * V + x];\n      if (p_out)"),
    "cdf_margin_not_over_R": ("*margin_out = (R > 0.0) ? fmin(m0, m1) / R : 0.0;",
                              "*margin_out = (R > 0.0) ? fmin(m0, m1) : 0.0;"),
    "acc_margin_past_n": ("      fprob += accept_flag_measure(p, q, window);\n      if (!(u * q < p)) { n = i; break; }",
                          "      fprob += accept_flag_measure(p, q, window);\n      if (!(u * q < p) && n == k) n = i;"),
    "flag_prob_without_cdf": ("      fprob += cdf_flag_measure(r, V, window, cb);\n",
                              "\n"),
    "claim_ignores_decisions": ("      if (accepted == claimed) continue;",
                                "      if (1) continue;"),
    "claim_interval_off_by_one": ("      for (int j = 0; j < t; ++j) c0 += w[j];",
                                  "      for (int j = 0; j <= t; ++j) c0 += w[j];"),
    "grow_gap_ignores_final_cut": ("    if (nn > M && M > 0) { double g = cut_gap(val, order, nn, M); if (g < gap) gap = g; }",
                                   "    (void)cut_gap;"),
    "grow_gap_counts_ties": ("  const double vk = val[order[keep - 1]], vd = val[order[keep]];\n  double g = INFINITY;",
                             "  const double vk = val[order[keep - 1]], vd = val[order[keep]];\n  double g = vk - vd;"),
    "f64_logits_read_as_f32": ("  if (dtype == OR_F64) return ((const double*)base)[idx];",
                               "  if (dtype == OR_F64) return (double)((const float*)base)[idx];"),
    "mask_wrong_word": ("        row[cur / 32] |= 1u << (cur % 32);\n        ++d;",
                        "        row[cur % W] |= 1u << (cur % 32);\n        ++d;"),
}


class _Variant:
    """Same API as the oracle module, bound to a mutated library."""

    OracleError = oracle.OracleError

    def __init__(self, lib):
        self.lib = lib

    def verify_sample(self, *a, **kw):
        return oracle.verify_sample(*a, lib=self.lib, **kw)

    def verify_greedy(self, *a, **kw):
        return oracle.verify_greedy(*a, lib=self.lib, **kw)

    def verify_tree_greedy(self, *a, **kw):
        return oracle.verify_tree_greedy(*a, lib=self.lib, **kw)

    def tree_mask(self, *a, **kw):
        return oracle.tree_mask(*a, lib=self.lib, **kw)

    def kv_commit(self, *a, **kw):
        return oracle.kv_commit(*a, lib=self.lib, **kw)

    def lm_head_greedy(self, *a, **kw):
        return oracle.lm_head_greedy(*a, lib=self.lib, **kw)

    def tree_grow(self, *a, **kw):
        return oracle.tree_grow(*a, lib=self.lib, **kw)

    def sample_claim(self, *a, **kw):
        return oracle.sample_claim(*a, lib=self.lib, **kw)

    def lm_head_sample(self, *a, **kw):
        return oracle.lm_head_sample(*a, lib=self.lib, **kw)

    def expected_tokens(self, *a, **kw):
        return oracle.expected_tokens(*a, lib=self.lib, **kw)

    def speedup_model(self, *a, **kw):
        return oracle.speedup_model(*a, lib=self.lib, **kw)


def _pin_checks(o):
    yield lambda: pins.test_worked_example_expected_tokens_and_speedup(o)
    yield lambda: pins.test_emission_law_equals_target_first_position(o, 1, 8, 0.7)
    yield lambda: pins.test_emission_law_equals_target_later_position(o, 4)
    yield lambda: pins.test_bonus_token_law_is_last_target_row(o, 3)
    yield lambda: pins.test_zero_probability_cases(o)
    yield lambda: pins.test_p_q_reported_for_every_row(o)
    yield lambda: pins.test_greedy_equals_argmax_decoding(o, "f32", 5)
    yield lambda: pins.test_tree_bruteforce(o, 1)
    yield lambda: pins.test_star_tree(o)
    yield lambda: pins.test_tree_mask_chain_is_causal(o)
    yield lambda: pins.test_tree_mask_equals_closure(o, 1)
    yield lambda: pins.test_kv_commit_equals_appending_the_path(o, 0)
    yield lambda: pins.test_kv_commit_chain_and_empty_paths_change_nothing(o)
    yield lambda: pins.test_lm_head_matches_float64_matmul(o)
    yield lambda: pins.test_lm_head_equals_unfused_greedy_on_exact_logits(o, 0)
    yield lambda: pins.test_lm_head_ties_and_subset(o)
    yield lambda: pins.test_tree_grow_one_layer_is_top_m_of_the_root_row(o)
    yield lambda: pins.test_tree_grow_worked_example_frontier_by_value(o)
    yield lambda: pins.test_tree_grow_ties_take_the_lower_token(o)
    yield lambda: pins.test_tree_grow_two_layers_full_expansion(o)
    yield lambda: pins.test_tree_grow_k1_is_the_greedy_chain(o)
    yield lambda: pins.test_tree_grow_structure(o, 0)
    yield lambda: pins.test_margins_and_flag_probability_worked_example(o)
    yield lambda: pins.test_claim_violation_worked_example(o)
    yield lambda: pins.test_tree_grow_min_gap_worked_example(o)
    yield lambda: pins.test_lm_head_sample_equals_plain_sampling_on_exact_logits(o)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mutated = tmp_path / f"mut_{name}.c"
    mutated.write_text(src.replace(old, new))
    lib_path = tmp_path / f"libmut_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib_path),
                    str(mutated), "-lm"], check=True)
    o = _Variant(oracle.load_variant(str(lib_path)))
    caught = []
    for check in _pin_checks(o):
        try:
            check()
        except (AssertionError, oracle.OracleError) as e:  # the pin fired
            caught.append(type(e).__name__)
            break
    assert caught, f"mutant {name} survived every pin"
