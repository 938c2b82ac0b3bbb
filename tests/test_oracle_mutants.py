"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle's C source (a
flipped sign, a transposed ratio, a dropped temperature, a wrong row index, a
non-strict comparison, a wrong bf16 shift, ...), compiles it on the CPU and
runs the pins that should notice: every mutant must fail at least one of them.
The committed oracle is never modified.
"""
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
import test_tree_pins as tpins
import test_row_sampler_pins as rpins
import test_tree_sample_pins as spins
import test_mtp_pins as mpins
import test_tree_builder_pins as bpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_oracle.c")

# (name, text in the source, replacement)
MUTANTS = [
    ("residual_sign", "double d = pj[v] - qj[v];", "double d = qj[v] - pj[v];"),
    ("residual_unclamped", "w[v] = d > 0.0 ? d : 0.0;", "w[v] = d;"),
    ("ratio_transposed", "double ratio = exp(((tx - mt) - (dx - md)) / T) * (Sd / St);",
     "double ratio = exp(((dx - md) - (tx - mt)) / T) * (St / Sd);"),
    ("ratio_sums_dropped", "double ratio = exp(((tx - mt) - (dx - md)) / T) * (Sd / St);",
     "double ratio = exp(((tx - mt) - (dx - md)) / T);"),
    ("draft_temperature_dropped", "softmax_row(draft, dtype, (size_t)b * K + i, V, T, q, &md, &Sd);",
     "softmax_row(draft, dtype, (size_t)b * K + i, V, 1.0, q, &md, &Sd);"),
    ("target_row_off_by_one", "softmax_row(target, dtype, (size_t)b * (K + 1) + i, V, T, p, &mt, &St);",
     "softmax_row(target, dtype, (size_t)b * (K + 1) + i + 1, V, T, p, &mt, &St);"),
    ("tail_from_row_zero", "softmax_row(target, dtype, (size_t)b * (K + 1) + j, V, T, pj, NULL, NULL);",
     "softmax_row(target, dtype, (size_t)b * (K + 1) + (j < K ? j : 0), V, T, pj, NULL, NULL);"),
    ("last_rejection_not_first", "j = i;\n                        decided = 1;", "j = i;"),
    ("inverse_cdf_not_strict", "if (C > target) {", "if (C >= target) {"),
    ("softmax_max_not_subtracted", "        p[v] = exp((logit_at(logits, dtype, off + v) - m) / T);",
     "        p[v] = exp(logit_at(logits, dtype, off + v) / T);"),
    ("acceptance_not_strict", "!((double)u_accept[(size_t)b * K + i] < thr)",
     "!((double)u_accept[(size_t)b * K + i] <= thr)"),
    ("greedy_out_of_range_token_accepted", "                    if (x != am) { j = i; break; }",
     "                    if (x != am && x >= 0) { j = i; break; }"),
    ("threshold_unclamped", "                        thr = ratio < 1.0 ? ratio : 1.0;", "                        thr = ratio;"),
    ("probs_p_and_q_swapped", "probs[((size_t)b * K + i) * 3 + 0] = px;", "probs[((size_t)b * K + i) * 3 + 0] = qx;"),
    ("extra_alone_greedy_row_off", "                bonus_token[b] = argmax_row(target, dtype, (size_t)b * (K + 1) + j, V);",
     "                bonus_token[b] = argmax_row(target, dtype, (size_t)b * (K + 1) + (j > 0 ? j - 1 : 0), V);"),
    ("extra_alone_length_past_k_accepted", "            if (j < 0 || j > K) {\n                bonus_token[b] = -1;",
     "            if (j < 0) {\n                bonus_token[b] = -1;"),
    ("vanished_residual_not_redrawn", "        if (W > 0.0) return inverse_cdf(w, V, u, lo, hi);",
     "        return inverse_cdf(w, V, u, lo, hi);"),
    ("tree_greedy_depth_off", "        while (depth < max_depth) {\n            int want",
     "        while (depth <= max_depth) {\n            int want"),
    ("tree_greedy_last_matching_child",
     "                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == want) {\n                    next = c;\n                    break;",
     "                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == want) {\n                    next = c;"),
    ("tree_sample_last_matching_child",
     "                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == draw[cur]) {\n                    next = c;\n                    break;",
     "                if (parents[c] == cur && node_tokens[(size_t)b * N + c] == draw[cur]) {\n                    next = c;"),
    ("tree_path_token_of_parent",
     "            ot[depth] = node_tokens[(size_t)b * N + next];\n            ++depth;\n            pn[depth] = next;\n            cur = next;\n        }\n        path_len[b] = depth;\n        ot[depth] = argmax_row",
     "            ot[depth] = node_tokens[(size_t)b * N + cur];\n            ++depth;\n            pn[depth] = next;\n            cur = next;\n        }\n        path_len[b] = depth;\n        ot[depth] = argmax_row"),
    ("residual_draft_row_off", "        softmax_row(draft, dtype, (size_t)b * K + j, V, T, qj, NULL, NULL);",
     "        softmax_row(draft, dtype, (size_t)b * K + (j + 1 < K ? j + 1 : j), V, T, qj, NULL, NULL);"),
    ("draft_logit_from_target", "double dx = logit_at(draft, dtype, ((size_t)b * K + i) * (size_t)V + x);",
     "double dx = logit_at(target, dtype, ((size_t)b * (K + 1) + i) * (size_t)V + x);"),
    ("uniform_of_position_zero", "!((double)u_accept[(size_t)b * K + i] < thr)", "!((double)u_accept[(size_t)b * K] < thr)"),
    ("emitted_counts_missing_extra", "            } else {\n                num_emitted[b] = j;\n            }",
     "            } else {\n                num_emitted[b] = j + 1;\n            }"),
    ("draft_token_of_next_position", "                    int x = draft_tokens[(size_t)b * K + i];\n                    double px",
     "                    int x = draft_tokens[(size_t)b * K + (i + 1 < K ? i + 1 : i)];\n                    double px"),
    ("tree_sample_node_token_of_parent",
     "            ot[depth] = node_tokens[(size_t)b * N + next];\n            ++depth;\n            pn[depth] = next;\n            cur = next;\n        }\n        path_len[b] = depth;\n        ot[depth] = draw[cur];",
     "            ot[depth] = node_tokens[(size_t)b * N + cur];\n            ++depth;\n            pn[depth] = next;\n            cur = next;\n        }\n        path_len[b] = depth;\n        ot[depth] = draw[cur];"),
    ("tree_sample_depth_off", "        while (depth < max_depth) {\n            int next = -1;",
     "        while (depth <= max_depth) {\n            int next = -1;"),
    ("rows_greedy_highest_index_on_ties", "            tokens[b] = argmax_row(logits, dtype, (size_t)b, V);",
     "            { int bb = 0; double bv = -INFINITY; for (int v = 0; v < V; ++v) { double l = logit_at(logits, dtype, "
     "(size_t)b * V + v); if (l >= bv) { bv = l; bb = v; } } tokens[b] = bb; }"),
    ("softmax_not_normalised", "    for (int v = 0; v < V; ++v) p[v] /= S;", "    for (int v = 0; v < V; ++v) p[v] /= 1.0;"),
    ("argmax_highest_index_on_ties", "if (l > bv) { bv = l; best = v; }", "if (l >= bv) { bv = l; best = v; }"),
    ("bf16_wrong_shift", "uint32_t w = ((uint32_t)h) << 16;", "uint32_t w = ((uint32_t)h) << 15;"),
    ("tree_extra_token_at_root", "ot[depth] = argmax_row(target, dtype, (size_t)b * N + cur, V);",
     "ot[depth] = argmax_row(target, dtype, (size_t)b * N + 0, V);"),
    ("tree_any_child", "if (parents[c] == cur && node_tokens[(size_t)b * N + c] == want)",
     "if (parents[c] >= 0 && node_tokens[(size_t)b * N + c] == want)"),
    ("tree_sample_temperature_dropped",
     "softmax_row(target, dtype, (size_t)b * N + n, V, T, p, NULL, NULL);",
     "softmax_row(target, dtype, (size_t)b * N + n, V, 1.0, p, NULL, NULL);"),
    ("tree_sample_uniform_of_root", "(double)u_nodes[(size_t)b * N + n]", "(double)u_nodes[(size_t)b * N]"),
    ("tree_sample_matches_root_draw", "node_tokens[(size_t)b * N + c] == draw[cur]",
     "node_tokens[(size_t)b * N + c] == draw[0]"),
    ("tree_sample_extra_is_argmax", "ot[depth] = draw[cur];",
     "ot[depth] = argmax_row(target, dtype, (size_t)b * N + cur, V);"),
    ("rows_temperature_dropped", "softmax_row(logits, dtype, (size_t)b, V, T, p, NULL, NULL);",
     "softmax_row(logits, dtype, (size_t)b, V, 1.0, p, NULL, NULL);"),
    ("rows_uniform_of_row_zero", "tokens[b] = inverse_cdf(p, V, (double)u[b], &lo, &hi);",
     "tokens[b] = inverse_cdf(p, V, (double)u[0], &lo, &hi);"),
    ("rows_greedy_from_row_zero", "tokens[b] = argmax_row(logits, dtype, (size_t)b, V);",
     "tokens[b] = argmax_row(logits, dtype, (size_t)0, V);"),
    ("mask_self_dropped", "mask[(size_t)i * W + cur / 32] |= 1u << (cur % 32);\n        while (cur != 0) {",
     "while (cur != 0) {"),
    ("mask_wrong_bit", "            mask[(size_t)i * W + cur / 32] |= 1u << (cur % 32);\n        }",
     "            mask[(size_t)i * W + cur / 32] |= 1u << ((cur + 1) % 32);\n        }"),
    ("mask_depth_off_by_one", "        depth[i] = d;", "        depth[i] = d + 1;"),
    ("mask_one_level_only", "            cur = par;\n            ++d;", "            cur = par;\n            ++d;\n            if (d > 1) break;"),
    ("tree_sample_row_of_root", "softmax_row(target, dtype, (size_t)b * N + n, V, T, p, NULL, NULL);",
     "softmax_row(target, dtype, (size_t)b * N, V, T, p, NULL, NULL);"),
    ("mtp_no_shift", "for (int i = 0; i < K; ++i) nx[i] = in[i + 1];", "for (int i = 0; i < K; ++i) nx[i] = in[i];"),
    ("mtp_shift_right", "for (int i = 0; i < K; ++i) nx[i] = in[i + 1];",
     "for (int i = 1; i <= K; ++i) nx[i] = in[i - 1];"),
    ("mtp_pad_first", "        nx[K] = pad;", "        nx[0] = pad;"),
    ("mtp_plug_one_short", "for (int i = 0; i < n; ++i) nx[i] = out_tokens[(size_t)b * W + i];",
     "for (int i = 0; i + 1 < n; ++i) nx[i] = out_tokens[(size_t)b * W + i];"),
    ("mtp_plug_one_place_late", "for (int i = 0; i < n; ++i) nx[i] = out_tokens[(size_t)b * W + i];",
     "for (int i = 0; i < n && i < K; ++i) nx[i + 1] = out_tokens[(size_t)b * W + i];"),
    ("mtp_length_without_extra", "        if (seq_lens) seq_lens[b] += n;", "        if (seq_lens) seq_lens[b] += n > 0 ? n - 1 : 0;"),
    ("mtp_plug_from_row_zero", "nx[i] = out_tokens[(size_t)b * W + i];", "nx[i] = out_tokens[i];"),
    ("builder_ties_to_deeper", "    if (ma != mb) return ma < mb;", "    if (ma != mb) return ma > mb;"),
    ("builder_ties_to_larger_rank", "        if (a[j] != b[j]) return a[j] < b[j];", "        if (a[j] != b[j]) return a[j] > b[j];"),
    ("builder_last_factor_dropped", "    for (int j = 0; j < m; ++j) v *= acc[(size_t)j * S + (path[j] - 1)];",
     "    for (int j = 0; j + 1 < m; ++j) v *= acc[(size_t)j * S + (path[j] - 1)];"),
    ("builder_heads_reversed", "    for (int j = 0; j < m; ++j) v *= acc[(size_t)j * S + (path[j] - 1)];",
     "    for (int j = 0; j < m; ++j) v *= acc[(size_t)(m - 1 - j) * S + (path[j] - 1)];"),
    ("builder_smallest_first", "if (!found || v > best_v ||", "if (!found || v < best_v ||"),
    ("builder_parent_is_root", "                    parents[r] = t;", "                    parents[r] = 0;"),
    ("builder_expected_len_first_level", "            e += path_product(acc, S, paths + (size_t)q * K, m);",
     "            e += path_product(acc, S, paths + (size_t)q * K, 1);"),
]


def _pin_suite(lib):
    """Run the pins against `lib`; return the names of those that failed."""
    failed = []
    checks = [
        ("distribution", lambda: pins.check_distribution_preserved(lib, 4, 2, 0.8, 9)),
        ("distribution_k1", lambda: pins.check_distribution_preserved(lib, 5, 1, 1.0, 10)),
        ("hand_example", lambda: pins.test_hand_worked_three_token_example(lib)),
        ("greedy_argmax", lambda: pins.test_greedy_equals_argmax_decoding(lib)),
        ("invariants", lambda: pins.test_invariants_random(lib, "f32")),
        ("zero_weight", lambda: pins.test_residual_zero_weight_token_never_drawn(lib)),
        ("bf16", lambda: pins.test_bf16_decoding_equals_fp32_values(lib)),
        ("spike", lambda: pins.test_spiked_constant_row_closed_form(lib, 1000, 5.0, 1.0)),
        ("strict", lambda: pins.check_strict_acceptance_at_an_exact_ratio(lib)),
        ("greedy_range", lambda: pins.check_greedy_rejects_an_out_of_range_token(lib)),
        ("extra_alone", lambda: pins.check_extra_token_alone_rows_and_lengths(lib)),
        ("vanished", lambda: pins.check_vanished_residual_draws_from_p(lib)),
        ("tree", lambda: _tree_check(lib)),
        ("tree_brute", lambda: tpins.check_tree_walk_brute_force(lib)),
        ("tree_duplicates", lambda: tpins.check_lowest_index_child_on_duplicate_tokens(lib)),
        ("tree_sample_freq", lambda: spins.check_draw_frequencies(lib, V=4, T=0.5, M=4000)),
        ("tree_sample_walk", lambda: spins.check_walk_brute_force(lib)),
        ("tree_sample_greedy", lambda: spins.check_dominant_logit_is_greedy(lib)),
        ("mask_chain", lambda: tpins.check_chain_mask_is_causal(lib)),
        ("mask_paths", lambda: tpins.check_mask_against_path_enumeration(lib)),
        ("rows_freq", lambda: rpins.check_frequencies(lib, V=5, T=0.7, M=5000)),
        ("rows_greedy", lambda: rpins.check_greedy_is_argmax(lib)),
        ("rows_scaling", lambda: rpins.check_temperature_scaling(lib)),
        ("mtp_single", lambda: mpins.check_hand_worked_single_token(lib)),
        ("mtp_k2", lambda: mpins.check_hand_worked_k2(lib)),
        ("mtp_align", lambda: mpins.check_alignment_with_decoded_sequences(lib)),
        ("mtp_shift", lambda: mpins.check_nothing_emitted_is_the_shift(lib)),
        ("mtp_range", lambda: mpins.check_counts_out_of_range(lib)),
        ("builder_count", lambda: bpins.check_post_node_count(lib)),
        ("builder_full", lambda: bpins.check_full_tree_counts(lib)),
        ("builder_brute", lambda: bpins.check_optimal_by_brute_force(lib, 2, 3, 4, 0)),
        ("builder_brute2", lambda: bpins.check_optimal_by_brute_force(lib, 3, 3, 5, 3)),
        ("builder_chain", lambda: bpins.check_chain_closed_form(lib)),
        ("builder_ties", lambda: bpins.check_exact_ties_order(lib)),
        ("builder_dominate", lambda: bpins.check_chosen_dominate_candidates(lib)),
    ]
    for name, fn in checks:
        try:
            fn()
        except Exception:  # a failed assertion, or a pin that cannot even read the mutant's output
            failed.append(name)
    return failed


def _tree_check(lib):
    rng = np.random.default_rng(5)
    B, V, N = 40, 10, 12
    parents = tpins._random_tree(rng, N)
    target = rng.standard_normal((B, N, V)).astype(np.float32)
    am = target.argmax(-1)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(N):
            ch = [c for c in range(N) if parents[c] == n]
            pool = list(rng.permutation(V))
            if ch and rng.random() < 0.8:
                pool.remove(am[b, n])
                pool.insert(0, am[b, n])
            for c, t in zip(ch, pool):
                tokens[b, c] = t
    r = oracle.verify_tree(target, parents, tokens, 5, lib=lib)
    for b in range(B):
        path, bonus = tpins._brute_force_walk(target[b], parents, tokens[b], 5)
        assert r["path_len"][b] == len(path) - 1
        assert r["out_tokens"][b, len(path) - 1] == bonus


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_unmutated_oracle_passes_suite(oracle_lib):
    assert _pin_suite(oracle_lib) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor must occur exactly once: %r" % old
    path = os.path.join(workdir, name + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(workdir, name + ".so")
    oracle.build(force=True, src=path, out=so)
    lib = oracle.load(so)
    failed = _pin_suite(lib)
    assert failed, "planted mistake %r passed every pin" % name
