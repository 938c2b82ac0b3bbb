"""Pins of the tree helpers and of the oracle's greedy tree walk.

"Speculative-Decoding / Medusa" blog:
  section 三 (Attention Tree) prints 4096 paths and 4680 nodes for K = 4 heads
  with top-8 candidates, from prod s_i and sum prod s_j (tests/golden);
  it describes verification as: take the target's choice at a node, look for
  it among the node's candidate children, continue along the matching child;
  section 四 defines E[L] as the sum, over the tree's nodes, of the product of
  per-head top-i accuracies, and grows the tree greedily to 64 nodes.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from workloads import make_tree, medusa_tree

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "medusa_tree_counts.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_cartesian_tree_counts_match_page():
    g = _golden()
    tree = medusa_tree.cartesian_tree([g["topk"]] * g["heads"])
    assert tree.n_nodes - 1 == g["nodes"]          # nodes below the root
    assert tree.n_paths() == g["paths"]


@pytest.mark.parametrize("sizes", [[2, 3], [3, 1, 2], [1, 1, 1, 1], [4, 2, 3, 2]])
def test_cartesian_counts_closed_form(sizes):
    tree = medusa_tree.cartesian_tree(sizes)
    assert tree.n_paths() == int(np.prod(sizes))
    assert tree.n_nodes - 1 == sum(int(np.prod(sizes[:i + 1])) for i in range(len(sizes)))
    assert all(0 <= p < c for c, p in enumerate(tree.parents) if c > 0)


def test_sparse_tree_has_page_node_count_and_is_topological():
    g = _golden()
    tree = medusa_tree.build_sparse_tree(4, 8, g["sparse_tree_nodes"], medusa_tree.synthetic_accuracy)
    assert tree.n_nodes == g["sparse_tree_nodes"]
    assert tree.parents[0] == -1
    assert all(0 <= p < c for c, p in enumerate(tree.parents) if c > 0)
    assert max(tree.depth) <= 4


def _all_closed_subsets(full_paths, size):
    """Every ancestor-closed set of `size` non-root paths of a full tree."""
    nonroot = [p for p in full_paths if p]
    for combo in itertools.combinations(nonroot, size):
        s = set(combo)
        if all(p[:-1] in s or len(p) == 1 for p in combo):
            yield combo


@pytest.mark.parametrize("K,s,n,seed", [(2, 3, 4, 0), (3, 2, 5, 1), (2, 4, 6, 2), (3, 3, 5, 3)])
def test_greedy_tree_is_optimal_by_brute_force(K, s, n, seed):
    rng = np.random.default_rng(seed)
    table = rng.uniform(0.05, 0.95, size=(K + 1, s + 1))
    acc = lambda k, i: table[k, i]                      # noqa: E731
    full = medusa_tree.cartesian_tree([s] * K)
    best = max(sum(medusa_tree.path_value(p, acc) for p in sub)
               for sub in _all_closed_subsets(full.paths, n))
    greedy = medusa_tree.build_sparse_tree(K, s, n + 1, acc)
    assert abs(medusa_tree.expected_accept_length(greedy, acc) - best) < 1e-12


def test_expected_length_formula_small_case():
    """Two heads, top-1 each: E[L] = a1 + a1 * a2 (section 四 with a single path)."""
    acc = lambda k, i: {1: 0.7, 2: 0.4}[k] if i == 1 else 0.0   # noqa: E731
    tree = medusa_tree.cartesian_tree([1, 1])
    assert abs(medusa_tree.expected_accept_length(tree, acc) - (0.7 + 0.7 * 0.4)) < 1e-15


# ------------------------------------------------------ oracle tree walk

def _random_tree(rng, N, max_children=4):
    parents = [-1]
    for c in range(1, N):
        parents.append(int(rng.integers(0, c)))
    return np.array(parents, np.int32)


def _brute_force_walk(target, parents, tokens, max_depth):
    """Longest root path whose every node carries argmax of its parent's row.

    With distinct tokens among siblings such a path is unique; found here by
    enumerating every root path of the tree."""
    N = len(parents)
    am = target.argmax(-1)
    paths = [[0]]
    frontier = [[0]]
    while frontier:
        nxt = []
        for path in frontier:
            for c in range(1, N):
                if parents[c] == path[-1]:
                    nxt.append(path + [c])
        paths += nxt
        frontier = nxt
    valid = [p for p in paths
             if len(p) - 1 <= max_depth and all(tokens[p[k + 1]] == am[p[k]] for k in range(len(p) - 1))]
    best = max(valid, key=len)
    return best, am[best[-1]]


def check_tree_walk_brute_force(lib=None, seed=21):
    rng = np.random.default_rng(seed)
    B, V = 60, 12
    for trial in range(8):
        N = int(rng.integers(1, 24))
        parents = _random_tree(rng, N)
        target = rng.standard_normal((B, N, V)).astype(np.float32)
        am = target.argmax(-1)
        tokens = np.zeros((B, N), np.int32)
        ch = [[c for c in range(N) if parents[c] == n] for n in range(N)]
        for b in range(B):
            for n in range(N):
                if not ch[n]:
                    continue
                pool = list(rng.permutation(V))
                if rng.random() < 0.7:     # one child carries the parent's argmax
                    pool.remove(am[b, n])
                    pool.insert(int(rng.integers(0, len(ch[n]))), am[b, n])
                for c, t in zip(ch[n], pool):
                    tokens[b, c] = t
        max_depth = int(rng.integers(0, 6))
        r = oracle.verify_tree(target, parents, tokens, max_depth, lib=lib)
        for b in range(B):
            path, bonus = _brute_force_walk(target[b], parents, tokens[b], max_depth)
            L = len(path) - 1
            assert r["path_len"][b] == L
            assert list(r["path_nodes"][b, :L + 1]) == path
            assert (r["path_nodes"][b, L + 1:] == -1).all()
            assert list(r["out_tokens"][b, :L]) == [tokens[b, n] for n in path[1:]]
            assert r["out_tokens"][b, L] == bonus
            assert (r["out_tokens"][b, L + 1:] == -1).all()


def test_chain_tree_equals_linear_greedy():
    """A chain (parents[c] = c - 1) is a linear draft: same accepted length and tokens."""
    rng = np.random.default_rng(22)
    B, K, V = 50, 6, 40
    target = rng.integers(-3, 4, (B, K + 1, V)).astype(np.float32)      # with ties
    am = target.argmax(-1)
    draft_tok = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    lin = oracle.verify_linear(target, None, draft_tok, None, np.zeros(B, np.float32), 0.0)
    parents = np.arange(-1, K, dtype=np.int32)
    node_tokens = np.concatenate([np.zeros((B, 1), np.int32), draft_tok], axis=1)
    tr = oracle.verify_tree(target, parents, node_tokens, K)
    np.testing.assert_array_equal(tr["path_len"], lin["accept_len"])
    np.testing.assert_array_equal(tr["out_tokens"], lin["out_tokens"])


def test_medusa_workload_mean_length_estimates_expected_length():
    """Mean accepted length over many sequences of the 64-node workload -> E[L]."""
    B = 3000
    d = make_tree(4, "cpu", B=B, V=48, seed=77)
    tree = d["tree"]
    el = medusa_tree.expected_accept_length(tree, medusa_tree.synthetic_accuracy)
    r = oracle.verify_tree(d["target"].numpy(), d["parents"].numpy(), d["node_tokens"].numpy(),
                           d["max_depth"])
    L = r["path_len"].astype(np.float64)
    se = L.std() / np.sqrt(B)
    assert abs(L.mean() - el) < 4.5 * se, (L.mean(), el, se)


# ------------------------------------------------------ tree attention mask
# Section 三: the tree is flattened into one sequence, and a mask modelled on
# the causal mask keeps tokens of different paths from attending to each other:
# row i of the mask holds node i and its ancestors, and nothing else.

def check_chain_mask_is_causal(lib):
    N = 70
    r = oracle.tree_mask(np.arange(-1, N - 1, dtype=np.int32), lib=lib)
    np.testing.assert_array_equal(oracle.mask_bits(r["mask"], N), np.tril(np.ones((N, N), np.uint8)))
    np.testing.assert_array_equal(r["depth"], np.arange(N))


def check_mask_against_path_enumeration(lib, seed=61):
    rng = np.random.default_rng(seed)
    for trial in range(10):
        N = int(rng.integers(1, 150))
        parents = _random_tree(rng, N)
        r = oracle.tree_mask(parents, lib=lib)
        m = oracle.mask_bits(r["mask"], N)
        for i in range(N):
            path = [i]
            while path[-1] != 0:
                path.append(int(parents[path[-1]]))
            want = np.zeros(N, np.uint8)
            want[path] = 1
            np.testing.assert_array_equal(m[i], want)
            assert r["depth"][i] == len(path) - 1
        assert not r["bad"]


def test_chain_mask_is_the_causal_mask(oracle_lib):
    check_chain_mask_is_causal(oracle_lib)


def test_mask_rows_are_root_paths(oracle_lib):
    check_mask_against_path_enumeration(oracle_lib)


def test_cartesian_tree_mask_counts():
    """Top-(s_1..s_K) Cartesian tree: every node's row holds depth + 1 bits; siblings never see each other."""
    tree = medusa_tree.cartesian_tree([3, 2, 2])
    par = np.array(tree.parents, np.int32)
    r = oracle.tree_mask(par)
    m = oracle.mask_bits(r["mask"], len(par))
    np.testing.assert_array_equal(m.sum(1), r["depth"] + 1)
    np.testing.assert_array_equal(r["depth"], np.array(tree.depth))
    for c in range(1, len(par)):
        for c2 in range(1, len(par)):
            if c != c2 and par[c] == par[c2]:
                assert m[c, c2] == 0


def test_bad_parent_is_reported():
    r = oracle.tree_mask(np.array([-1, 0, 5, 1], np.int32))
    assert r["bad"]
    assert r["depth"][3] == 2 and r["depth"][2] == 0
    # a node that is its own parent stops its walk too (a parent must precede its child)
    r = oracle.tree_mask(np.array([-1, 0, 2, 2], np.int32))
    assert r["bad"] and r["depth"][2] == 0 and r["depth"][3] == 1


def test_tree_walk_matches_brute_force(oracle_lib):
    check_tree_walk_brute_force(oracle_lib)


def check_lowest_index_child_on_duplicate_tokens(lib):
    """When several children carry the target's choice, the walk takes the lowest-index one,
    greedy and sampled (with a dominant logit every draw is the argmax)."""
    # root 0 -> children 1, 2, 3 all carrying token 4 (the root's argmax); 1 -> 4, 2 -> 5, 3 -> 6
    parents = np.array([-1, 0, 0, 0, 1, 2, 3], np.int32)
    V = 8
    target = np.zeros((1, 7, V), np.float32)
    target[0, 0, 4] = 60.0                       # root: argmax 4
    target[0, 1:, 6] = 60.0                      # every other node: argmax 6
    tokens = np.array([[0, 4, 4, 4, 6, 6, 6]], np.int32)
    g = oracle.verify_tree(target, parents, tokens, 3, lib=lib)
    assert list(g["path_nodes"][0]) == [0, 1, 4, -1] and list(g["out_tokens"][0]) == [4, 6, 6, -1]
    u = np.full((1, 7), 0.5, np.float32)
    s = oracle.verify_tree_sample(target, parents, tokens, u, 1.0, 3, lib=lib)
    assert list(s["path_nodes"][0]) == [0, 1, 4, -1] and list(s["out_tokens"][0]) == [4, 6, 6, -1]
    # max_depth stops the walk even when a child would match
    g1 = oracle.verify_tree(target, parents, tokens, 1, lib=lib)
    assert list(g1["path_nodes"][0]) == [0, 1] and list(g1["out_tokens"][0]) == [4, 6]


def test_lowest_index_child_on_duplicate_tokens(oracle_lib):
    check_lowest_index_child_on_duplicate_tokens(oracle_lib)
