"""The pins bite: plant a plausible mistake in a copy of the oracle (on the CPU),
rebuild it, and check that at least one pin fails.  Each mutation names the
passage it breaks."""
import ctypes as C
import os
import subprocess

import pytest

import oracle as ORC

from . import test_oracle_ngram as TN
from . import test_oracle_ngram_fill as TF
from . import test_oracle_philox as TP
from . import test_oracle_price as TPR
from . import test_oracle_budget as TBU
from . import test_oracle_draft_sampling as TDS
from . import test_oracle_tree as TT
from . import test_oracle_tree_build as TB
from . import test_oracle_verify as TV

SRC = os.path.join(os.path.dirname(ORC.__file__), "spec_oracle.c")

MUTATIONS = [
    # (name, original text, mutated text, pins expected to catch it)
    ("philox multiplier", "#define PHILOX_M0 0xD2511F53u", "#define PHILOX_M0 0xD2511F55u",
     [TP.test_philox_known_answers]),
    ("philox key schedule", "k1 += PHILOX_W1;", "k1 += PHILOX_W0;", [TP.test_philox_known_answers]),
    ("uniform conversion", "(double)(w >> 8) * (1.0 / 16777216.0)", "(double)(w >> 9) * (1.0 / 16777216.0)",
     [TP.test_uniform_conversion_is_exact_24_bit]),
    ("n-gram tie to the oldest occurrence", "(l == best_l && j > best_j)", "(l == best_l && j < best_j)",
     [TN.test_runner_up_with_different_follower_disagrees]),
    ("n-gram agreement compares the wrong tokens", "x[second_j + 1] == x[best_j + 1]",
     "x[second_j] == x[best_j]", [TN.test_runner_up_with_different_follower_disagrees]),
    ("n-gram continuation off by one", "x[best_j + 1 + i]", "x[best_j + i]",
     [TN.test_exact_copy_gives_its_continuation]),
    ("n-gram ignores the cap", "int32_t limit = copy_cap < j + 1 ? copy_cap : j + 1;",
     "int32_t limit = j + 1;", [TN.test_match_length_capped_at_n_max_and_copy_length_at_cap]),
    ("Eq. (1) drops the agreement term", "z = z + e->delta * (double)a;", "z = z;",
     [TPR.test_full_match_indicator_and_agreement_terms]),
    ("Eq. (1) swaps first / later copy weights", "(first ? e->kappa_first : e->kappa_rest)",
     "(first ? e->kappa_rest : e->kappa_first)",
     [TPR.test_copy_length_term_adds_5_7_logits_at_the_first_position]),
    ("Eq. (1) drops the 1/15 in the log", "log((double)mm / (double)e->m_ref)", "log((double)mm)",
     [TPR.test_full_match_indicator_and_agreement_terms]),
    ("Eq. (1) sign of the match-length term", "z = z + (first ? e->w_first : e->w_rest) * (double)(n - e->n_ref);",
     "z = z - (first ? e->w_first : e->w_rest) * (double)(n - e->n_ref);",
     [TPR.test_full_match_indicator_and_agreement_terms]),
    ("Eq. (3) sign of the price", "float t = S[k] - lambda;", "float t = S[k] + lambda;",
     [TPR.test_table8_chain_values]),
    ("contains rule takes the min", "Sr[k] = Sg[k] > Sd[k] ? Sg[k] : Sd[k];", "Sr[k] = Sg[k] < Sd[k] ? Sg[k] : Sd[k];",
     [TPR.test_contains_rule_merges_survivals_and_continues_with_h]),
    ("value rule ties to the model chain", "oracle_chain_value(Sg, gl, lambda) >=",
     "oracle_chain_value(Sg, gl, lambda) >", [TPR.test_value_rule_ties_go_to_the_ngram_chain]),
    ("allocation ties to the higher request", "if (a->r != b->r) return a->r < b->r ? -1 : 1;",
     "if (a->r != b->r) return a->r > b->r ? -1 : 1;", [TPR.test_allocation_ties_go_to_lower_request_then_position]),
    ("allocation keeps the lowest survivals", "if (a->s > b->s) return -1; /* survival descending */",
     "if (a->s > b->s) return 1; /* survival descending */",
     [TPR.test_allocation_is_the_best_prefix_closed_set_brute_force]),
    ("row offsets forget the bonus row", "row_off[r + 1] = row_off[r] + verify_len[r] + 1;",
     "row_off[r + 1] = row_off[r] + verify_len[r];", [TPR.test_allocation_is_the_best_prefix_closed_set_brute_force]),
    ("accept ratio inverted", "ratio = p[yi] / q[yi];", "ratio = q[yi] / p[yi];",
     [lambda o: TV.test_lossless_with_probabilistic_drafts(o, 3, 2, 0.7, 1)]),
    ("residual max(0, q - p)", "v = p[x] - q[x] > 0.0 ? p[x] - q[x] : 0.0;", "v = q[x] - p[x] > 0.0 ? q[x] - p[x] : 0.0;",
     [lambda o: TV.test_lossless_with_probabilistic_drafts(o, 3, 2, 0.7, 1)]),
    ("point-mass residual keeps the rejected token", "v = (x == y) ? 0.0 : p[x];", "v = p[x];",
     [lambda o: TV.test_lossless_with_point_mass_drafts(o, 3, 2, 1.0, 4)]),
    ("bonus drawn from the last draft row", "row_softmax(target_logits, (int64_t)base + ell, vocab, dtype, temperature, p);",
     "row_softmax(target_logits, (int64_t)base + ell - (ell > 0), vocab, dtype, temperature, p);",
     [lambda o: TV.test_lossless_with_point_mass_drafts(o, 3, 2, 1.0, 4)]),
    ("temperature ignored", "p[x] = exp((logit_at(base, row * vocab + x, dtype) - m) / T);",
     "p[x] = exp((logit_at(base, row * vocab + x, dtype) - m));",
     [lambda o: TV.test_lossless_with_point_mass_drafts(o, 4, 3, 0.7, 5)]),
    ("inverse CDF one token late", "if (run > t) return x;", "if (run > t) return x + (x + 1 < vocab);",
     [TV.test_bonus_draws_follow_p_chi_square]),
    ("greedy ties to the highest index", "if (best < 0 || z > bv) {", "if (best < 0 || z >= bv) {",
     [TV.test_greedy_ties_go_to_the_lowest_index]),
    ("tree walk reads the child's own row", "a = row_argmax(logits, (int64_t)base + cur, vocab, dtype);",
     "a = row_argmax(logits, (int64_t)base + (cur > 0 ? parent[base + cur] : 0), vocab, dtype);",
     [TT.test_path_by_brute_force_over_root_to_node_paths]),
    ("tree commits the last path token, not its argmax", "out_tokens[(int64_t)r * max_nodes + len - 1] = a;",
     "out_tokens[(int64_t)r * max_nodes + len - 1] = tok[base + cur];",
     [TT.test_path_by_brute_force_over_root_to_node_paths]),
    # candidate-tree builder (AdaSpark sec. 2.2, sec. 3.1, sec. 3.3 Eq. (6))
    ("tree builder drops the none outcome of Eq. (6)", "double den = 1.0;", "double den = 0.0;",
     [TB.test_chain_only_tree_is_a_path_of_sigmoids, lambda o: TB.test_equal_scores_share_one_softmax_with_none(o, 4, -1.3)]),
    ("tree builder ties to the higher index", "while (at > 0 && (Q[order[at - 1]] < Q[j])) --at;",
     "while (at > 0 && (Q[order[at - 1]] <= Q[j])) --at;", [TB.test_ties_go_to_the_lower_index]),
    ("tree builder rewards contradicted candidates", "(contra[j] ? -adj : 0.0)", "(contra[j] ? adj : 0.0)",
     [TB.test_ngram_chain_agrees_with_picks_then_extends,
      TB.test_ngram_chain_that_matches_no_candidate_contradicts_them_all]),
    ("tree builder hangs siblings under their own pick",
     "cpar[j] = (i == 0) ? 0 : 1 + (i - 1) * Kc;",
     "cpar[j] = (k == 0) ? ((i == 0) ? 0 : 1 + (i - 1) * Kc) : 1 + i * Kc;",
     [TB.test_picks_form_a_spine_and_siblings_are_leaves]),
    ("tree builder lays children out in decreasing index",
     "for (int32_t c = N - 1; c > j; --c) /* pushed", "for (int32_t c = j + 1; c < N; ++c) /* pushed",
     [lambda o: TB.test_layout_is_depth_first_with_children_in_index_order(o, 0),
      lambda o: TB.test_layout_is_depth_first_with_children_in_index_order(o, 1)]),
    ("tree builder multiplies Q by the parent's q", "for (int32_t j = 1; j < N; ++j) Q[j] = Q[cpar[j]] * q[j];",
     "for (int32_t j = 1; j < N; ++j) Q[j] = Q[cpar[j]] * q[cpar[j] > 0 ? cpar[j] : j];",
     [TB.test_chain_only_tree_is_a_path_of_sigmoids, TB.test_ngram_chain_agrees_with_picks_then_extends]),
    ("tree builder duplicates an n-gram node another chain made", "        if (old >= 0) {\n          cur = old;",
     "        if (0) {\n          cur = old;", [TB.test_chains_from_picks_share_their_nodes]),
    ("tree builder lets a contradiction beat an agreement", "agreed[j] ? adj : (contra[j] ? -adj : 0.0)",
     "contra[j] ? -adj : (agreed[j] ? adj : 0.0)",
     [TB.test_a_candidate_agreed_by_one_chain_and_contradicted_by_another_is_agreed]),
    ("tree builder starts a pick's chain below the wrong pick", "int32_t cur = (ch == 0) ? 0 : 1 + (ch - 1) * Kc;",
     "int32_t cur = (ch == 0) ? 0 : 1 + ch * Kc;",
     [TB.test_chains_from_picks_share_their_nodes,
      TB.test_a_candidate_agreed_by_one_chain_and_contradicted_by_another_is_agreed]),
    # n-gram fill of the tree (AdaSpark sec. 2.2, sec. 3.3)
    ("fill ties to the oldest occurrence", "(l == top_l && j > top_j)", "(l == top_l && j < top_j)",
     [TF.test_equal_matches_go_to_the_most_recent]),
    ("fill does not read on along the passage", "q = top_j + 2;", "q = -1;",
     [TF.test_the_passage_is_read_on_even_where_a_new_lookup_would_leave_it]),
    ("fill follower by recency only", "                  ++cnt;\n", "                  cnt = 1;\n",
     [TF.test_follower_fallback_takes_the_most_frequent]),
    ("fill follower ties to the oldest", "(cnt == best_cnt && last > best_last)", "(cnt == best_cnt && last < best_last)",
     [TF.test_follower_ties_go_to_the_most_recent]),
    ("fill counts followers of two tokens", "if (x[i - 2] == a && x[i - 1] == b && x[i] == d && x[i + 1] == f) {",
     "if (x[i - 1] == b && x[i] == d && x[i + 1] == f) {",
     [lambda o, s=s: TF.test_every_token_is_backed_by_its_evidence(o, s, 4, 5, 0.0) for s in range(4)]),
    ("fill depth counted from the chain's start", "int32_t cap = max_depth - c;", "int32_t cap = max_depth;",
     [TF.test_depth_limit_counts_from_the_anchor]),
    ("fill forgets the picks on the path", "for (int32_t i = 0; i < c; ++i) ext[m++]",
     "for (int32_t i = 0; i < 0; ++i) ext[m++]", [TF.test_chain_from_a_pick_continues_the_pick]),
    ("fill passage overruns the text", "if (q >= 0 && q <= T - 1) {", "if (q >= 0 && q <= T) {",
     [TF.test_chain_reads_along_an_earlier_passage]),
    # budget sizing (Hybrid Spark sec. 2, sec. 4.3 Eq. (2), App. F)
    ("budget forgets the one token every request emits", "double A = (double)batch, best = A / C0;",
     "double A = 0.0, best = A / C0;", [lambda o: TBU.test_budget_against_exact_rationals(o, 3)]),
    ("budget ties to the larger b", "    if (G > best) {\n      best = G;\n      bs = b;",
     "    if (G >= best) {\n      best = G;\n      bs = b;", [lambda o: TBU.test_equal_survivals_closed_form(o, 0.5, 8.0, 1.0)]),
    ("budget counts slots past max_verify_len",
     "int32_t len = chain_len[r] < max_verify_len ? chain_len[r] : max_verify_len;",
     "int32_t len = chain_len[r];", [TBU.test_only_verifiable_slots_count]),
    ("budget takes the smallest survivals first", "return (x < y) - (x > y);", "return (x > y) - (x < y);",
     [lambda o: TBU.test_slot_price_rule_of_eq_2(o, 0)]),
    # probabilistic drafting (Hybrid Spark sec. 4.5, App. H)
    ("drafts draw with verification's counters", "0x40000000u + (uint32_t)k, (uint32_t)step",
     "(uint32_t)k, (uint32_t)step", [TDS.test_uniform_counter_domain]),
    ("drafts ignore the temperature", "row_softmax(draft_logits, row, vocab, dtype, temperature, q);",
     "row_softmax(draft_logits, row, vocab, dtype, 1.0, q);",
     [lambda o: TDS.test_temperature_half_squares_the_odds(o, 0.08, 1)]),
]


@pytest.fixture(scope="module")
def src_text():
    return open(SRC).read()


@pytest.mark.parametrize("name,orig,mut,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, src_text, name, orig, mut, pins):
    assert src_text.count(orig) == 1, f"mutation anchor not unique: {orig!r}"
    src = tmp_path / "spec_oracle.c"
    src.write_text(src_text.replace(orig, mut))
    hdr = os.path.join(os.path.dirname(SRC), "spec_oracle.h")
    (tmp_path / "spec_oracle.h").write_text(open(hdr).read())
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(src), "-lm"])
    ORC.lib()
    saved = ORC._lib
    mut_lib = C.CDLL(str(so))
    ORC._declare(mut_lib)
    ORC._lib = mut_lib
    try:
        caught = 0
        for pin in pins:
            try:
                pin(ORC)
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin caught the planted mistake: {name}"
    finally:
        ORC._lib = saved
