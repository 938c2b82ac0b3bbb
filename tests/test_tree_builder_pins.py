"""Pins of the oracle's greedy sparse-tree builder.

"Speculative-Decoding / Medusa" blog, section 四 (optimized tree
construction): with a_k^(i) the accuracy of head k's i-th ranked token, taken
as independent, a node's path [i_1..i_m] is accepted with probability
prod_j a_j^(i_j); E[L] sums that product over the tree's nodes; the tree is
grown one node at a time by the candidate of largest product, to a fixed node
count (64 nodes in the post).  Section 三 gives the full tree's counts,
prod s_i paths and sum prod s_j nodes (tests/golden).

The pins: the post's 64-node count; the full tree's closed-form counts; E[L]
equals the best ancestor-closed node set found by brute force; a chain's E[L]
in closed form; a hand-derived order under exact ties; every chosen node's
product is at least every unchosen candidate's.
"""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "medusa_tree_counts.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def _synthetic(K, S):
    return np.array([[0.6 * 0.8 ** k * 0.5 ** i for i in range(1, S + 1)] for k in range(1, K + 1)])


def _paths(r):
    """Rank path of every node, rebuilt from parents and ranks."""
    out = []
    for c in range(len(r["parents"])):
        p = () if c == 0 else out[r["parents"][c]] + (int(r["rank"][c]),)
        out.append(p)
    return out


def _value(acc, path):
    v = 1.0
    for j, i in enumerate(path):
        v *= acc[j, i - 1]
    return v


def check_post_node_count(lib):
    g = _golden()
    r = oracle.build_sparse_tree(_synthetic(g["heads"], g["topk"]), g["sparse_tree_nodes"], lib=lib)
    n = len(r["parents"])
    assert n == g["sparse_tree_nodes"] and r["parents"][0] == -1
    assert all(0 <= r["parents"][c] < c for c in range(1, n))
    assert all(r["depth"][c] == r["depth"][r["parents"][c]] + 1 for c in range(1, n))
    assert r["depth"].max() <= g["heads"] and r["rank"].max() <= g["topk"]


def check_full_tree_counts(lib, K=3, S=4):
    r = oracle.build_sparse_tree(np.full((K, S), 0.5), 10 ** 4, lib=lib)
    n = len(r["parents"])
    assert n - 1 == sum(S ** m for m in range(1, K + 1))            # sum_i prod_{j<=i} s_j nodes
    has_child = np.zeros(n, bool)
    has_child[r["parents"][1:]] = True
    assert int((~has_child).sum()) == S ** K                         # prod s_i root-to-leaf paths


def check_optimal_by_brute_force(lib, K, S, n, seed):
    rng = np.random.default_rng(seed)
    acc = rng.uniform(0.05, 0.95, size=(K, S))
    full = [p for m in range(1, K + 1) for p in itertools.product(range(1, S + 1), repeat=m)]
    best = 0.0
    for combo in itertools.combinations(full, n):
        s = set(combo)
        if all(len(p) == 1 or p[:-1] in s for p in combo):
            best = max(best, sum(_value(acc, p) for p in combo))
    r = oracle.build_sparse_tree(acc, n + 1, lib=lib)
    assert abs(r["expected_len"] - best) < 1e-12
    assert abs(sum(_value(acc, p) for p in _paths(r)[1:]) - r["expected_len"]) < 1e-12


def check_chain_closed_form(lib):
    acc = np.array([[0.9], [0.7], [0.4], [0.2]])
    r = oracle.build_sparse_tree(acc, 5, lib=lib)
    assert r["parents"].tolist() == [-1, 0, 1, 2, 3] and r["rank"].tolist() == [0, 1, 1, 1, 1]
    assert abs(r["expected_len"] - (0.9 + 0.9 * 0.7 + 0.9 * 0.7 * 0.4 + 0.9 * 0.7 * 0.4 * 0.2)) < 1e-15


def check_exact_ties_order(lib):
    # every accuracy 1/2: (1) and (2) tie at 1/2 -> (1) first; then (2); then the four depth-2 paths tie at 1/4
    r = oracle.build_sparse_tree(np.full((2, 2), 0.5), 5, lib=lib)
    assert _paths(r) == [(), (1,), (2,), (1, 1), (1, 2)]
    assert r["parents"].tolist() == [-1, 0, 0, 1, 1] and r["depth"].tolist() == [0, 1, 1, 2, 2]
    assert r["expected_len"] == 0.5 + 0.5 + 0.25 + 0.25
    # a tie across depths: (2) = 1/4 and (1, 1) = (1, 2) = 1/2 * 1/2 -> the shallower (2) first
    r = oracle.build_sparse_tree(np.array([[0.5, 0.25], [0.5, 0.5]]), 4, lib=lib)
    assert _paths(r) == [(), (1,), (2,), (1, 1)]


def check_chosen_dominate_candidates(lib, seed=11):
    rng = np.random.default_rng(seed)
    acc = np.sort(rng.uniform(0.01, 0.9, size=(4, 6)), axis=1)[:, ::-1].copy()
    r = oracle.build_sparse_tree(acc, 30, lib=lib)
    paths = _paths(r)
    chosen = set(paths)
    worst = min(_value(acc, p) for p in paths[1:])
    for p in paths:
        if len(p) < 4:
            for i in range(1, 7):
                c = p + (i,)
                if c not in chosen:
                    assert _value(acc, c) <= worst


def test_post_node_count(oracle_lib):
    check_post_node_count(oracle_lib)


def test_full_tree_counts(oracle_lib):
    check_full_tree_counts(oracle_lib)
    check_full_tree_counts(oracle_lib, K=2, S=7)


@pytest.mark.parametrize("K,S,n,seed", [(2, 3, 4, 0), (3, 2, 5, 1), (2, 4, 6, 2), (3, 3, 5, 3)])
def test_optimal_by_brute_force(oracle_lib, K, S, n, seed):
    check_optimal_by_brute_force(oracle_lib, K, S, n, seed)


def test_chain_closed_form(oracle_lib):
    check_chain_closed_form(oracle_lib)


def test_exact_ties_order(oracle_lib):
    check_exact_ties_order(oracle_lib)


def test_chosen_dominate_candidates(oracle_lib):
    check_chosen_dominate_candidates(oracle_lib)


def test_equals_the_workload_generator(oracle_lib):
    """The input generator's own (heap-based) builder gives the same 64-node tree."""
    from workloads import medusa_tree
    t = medusa_tree.build_sparse_tree(4, 8, 64, medusa_tree.synthetic_accuracy)
    acc = np.array([[medusa_tree.synthetic_accuracy(k, i) for i in range(1, 9)] for k in range(1, 5)])
    r = oracle.build_sparse_tree(acc, 64, lib=oracle_lib)
    assert r["parents"].tolist() == t.parents and r["rank"].tolist() == t.rank
