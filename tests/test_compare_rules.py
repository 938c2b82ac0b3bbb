"""The comparison rules that decide GPU-vs-oracle parity, on constructed results.

A mismatch is forgiven only as a counted near tie: the uniform lies within
NEAR_TIE of the boundary that decided it (the acceptance threshold, or an end
of the drawn token's cumulative interval).  Everything else must be equal.
These cases check that the rules forgive exactly that and catch the rest.
"""
import numpy as np

from oracle import compare


def _linear_oracle(accept_len, out_tokens, probs, cdf):
    return dict(accept_len=np.array(accept_len, np.int32), out_tokens=np.array(out_tokens, np.int32),
                num_emitted=np.array(accept_len, np.int32) + 1, probs=np.array(probs, np.float64),
                bonus_cdf=np.array(cdf, np.float64))


def _gpu(accept_len, out_tokens, probs):
    return dict(accept_len=np.array(accept_len, np.int32), out_tokens=np.array(out_tokens, np.int32),
                num_emitted=np.array(accept_len, np.int32) + 1, probs=np.array(probs, np.float32))


# one sequence, K = 2: oracle accepts x_0 = 5, rejects at position 1, extra token 9 in [0.3, 0.4)
ORA = _linear_oracle([1], [[5, 9, -1]], [[[0.2, 0.1, 1.0], [0.1, 0.3, 0.333]]], [[0.3, 0.4]])
PROBS = [[[0.2, 0.1, 1.0], [0.1, 0.3, 0.333]]]


def test_equal_results_are_exact():
    rep = compare.compare_linear(_gpu([1], [[5, 9, -1]], PROBS), ORA, [[0.5, 0.9]], [0.35], 1.0)
    assert rep.ok and rep.exact == 1


def test_acceptance_flip_is_a_tie_only_at_the_threshold():
    g = _gpu([2], [[5, 7, 3]], PROBS)          # the GPU accepted position 1 as well
    near = compare.compare_linear(g, ORA, [[0.5, 0.333 + 5e-7]], [0.35], 1.0)
    assert near.ok and near.accept_ties == 1
    far = compare.compare_linear(g, ORA, [[0.5, 0.9]], [0.35], 1.0)
    assert not far.ok


def test_extra_token_flip_is_a_tie_only_at_an_interval_end():
    g = _gpu([1], [[5, 8, -1]], PROBS)          # a neighbouring extra token
    near = compare.compare_linear(g, ORA, [[0.5, 0.9]], [0.3 + 2e-7], 1.0)
    assert near.ok and near.bonus_ties == 1
    far = compare.compare_linear(g, ORA, [[0.5, 0.9]], [0.35], 1.0)
    assert not far.ok


def test_probability_tolerance():
    off = [[[0.2 + 2e-5, 0.1, 1.0], [0.1, 0.3, 0.333]]]
    rep = compare.compare_linear(_gpu([1], [[5, 9, -1]], off), ORA, [[0.5, 0.9]], [0.35], 1.0)
    assert not rep.ok
    ok = [[[0.2 + 5e-6, 0.1, 1.0], [0.1, 0.3, 0.333]]]
    assert compare.compare_linear(_gpu([1], [[5, 9, -1]], ok), ORA, [[0.5, 0.9]], [0.35], 1.0).ok


def test_greedy_forgives_nothing():
    ora = _linear_oracle([1], [[5, 9, -1]], np.zeros((1, 2, 3)), [[0.0, 0.0]])
    g = _gpu([1], [[5, 8, -1]], np.zeros((1, 2, 3)))
    assert not compare.compare_linear(g, ora, None, None, 0.0, check_probs=False).ok


def _tree(path_len, nodes, tokens):
    return dict(path_len=np.array(path_len, np.int32), path_nodes=np.array(nodes, np.int32),
                out_tokens=np.array(tokens, np.int32))


def test_sampled_tree_tie_only_on_a_path_node():
    ora = _tree([1], [[0, 2, -1]], [[4, 6, -1]])
    ora["node_cdf"] = np.zeros((1, 4, 2))
    ora["node_cdf"][0, 2] = [0.5, 0.6]          # the draw at node 2 made the extra token 6
    ora["node_cdf"][0, 3] = [0.1, 0.2]
    g = _tree([1], [[0, 2, -1]], [[4, 7, -1]])
    u = np.array([[0.9, 0.9, 0.6 - 3e-7, 0.1 + 3e-7]])
    near = compare.compare_tree_sample(g, ora, u)
    assert near.ok and near.bonus_ties == 1
    # a uniform near a boundary at node 3, which is on neither path, forgives nothing
    u2 = np.array([[0.9, 0.9, 0.55, 0.1 + 3e-7]])
    assert not compare.compare_tree_sample(g, ora, u2).ok
    assert compare.compare_tree_sample(_tree([1], [[0, 2, -1]], [[4, 6, -1]]), ora, u2).exact == 1


def test_sampled_tree_tie_only_at_the_node_where_the_walks_part():
    """The walks share the root and node 1, then part: only node 1's draw may be a near tie.
    A uniform at the root that sits on an interval edge, where the walks agreed, forgives
    nothing (the looser rule counted any node on either path)."""
    ora = _tree([2], [[0, 1, 5, -1]], [[10, 11, 12, -1]])
    ora["node_cdf"] = np.zeros((1, 8, 2))
    ora["node_cdf"][0, 0] = [0.3, 0.4]
    ora["node_cdf"][0, 1] = [0.7, 0.8]
    g = _tree([1], [[0, 1, -1, -1]], [[10, 13, -1, -1]])   # at node 1 the GPU drew a token no child carries
    assert compare.compare_tree_sample(g, ora, np.array([[0.35, 0.8 - 2e-7, 0, 0, 0, 0, 0, 0]])).bonus_ties == 1
    rep = compare.compare_tree_sample(g, ora, np.array([[0.3 + 1e-7, 0.75, 0, 0, 0, 0, 0, 0]]))
    assert not rep.ok and "part at node 1" in rep.failures[0]
    # the GPU walk goes further than the oracle's: the last shared node decides
    g2 = _tree([3], [[0, 1, 5, 6]], [[10, 11, 12, 14]])
    ora2 = dict(ora, path_len=np.array([2], np.int32))
    ora2["node_cdf"][0, 5] = [0.2, 0.25]
    assert compare.compare_tree_sample(g2, ora2, np.array([[0.5, 0.5, 0, 0, 0, 0.25 - 1e-7, 0, 0]])).bonus_ties == 1
    assert not compare.compare_tree_sample(g2, ora2, np.array([[0.5, 0.7 + 1e-7, 0, 0, 0, 0.22, 0, 0]])).ok


def test_every_report_is_logged_with_its_label():
    compare.LABEL[0] = "unit-test-label"
    n = len(compare.LOG)
    ora = _tree([0], [[0, -1]], [[3, -1]])
    compare.compare_tree(ora, ora)
    assert len(compare.LOG) == n + 1 and compare.LOG[-1][0] == "unit-test-label" and compare.LOG[-1][1] == "tree"
    compare.LOG.pop()
