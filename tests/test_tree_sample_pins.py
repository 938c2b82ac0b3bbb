"""Pins of the oracle's tree walk in sampling mode.

"Speculative-Decoding / Medusa" blog, section 三 (Attention Tree): at a node
the target makes its choice, greedy or sampled, and verification continues
along the candidate child that carries it.  Sampled, the choice at node n is a
draw from softmax(target_n / T); the draw here is by inverse CDF with the
caller's uniform u[b, n] (the first v whose cumulative probability exceeds u).

The pins fix it against what the mathematics fixes:
  - over a fine grid of uniforms, each token is drawn with frequency p_v of
    the temperature softmax (the inverse CDF of a known distribution);
  - on random trees, the path equals a brute-force search over every root
    path, using draws made here from the definition;
  - with one dominant logit per row every draw is the argmax, and the walk
    reduces to the greedy walk.
"""
import numpy as np
import pytest

import oracle
import test_tree_pins as tpins


def _softmax64(row, T):
    x = row.astype(np.float64) / T
    e = np.exp(x - x.max())
    return e / e.sum()


def _draw(row, T, u):
    """First v whose cumulative probability exceeds u, and u's distance to the nearest boundary."""
    c = np.cumsum(_softmax64(row, T))
    target = float(u) * c[-1]
    v = int(np.searchsorted(c, target, side="right"))
    v = min(v, len(c) - 1)
    return v, float(np.min(np.abs(c / c[-1] - float(u))))


def check_draw_frequencies(lib, V=5, T=0.6, M=20000, seed=3):
    """Single-node trees: the draw at u_i = (i + 1/2) / M has frequency p_v to within 1/M."""
    rng = np.random.default_rng(seed)
    row = (rng.standard_normal(V) * 2.0).astype(np.float32)
    target = np.broadcast_to(row, (M, 1, V)).copy()
    u = ((np.arange(M) + 0.5) / M).astype(np.float32).reshape(M, 1)
    r = oracle.verify_tree_sample(target, np.array([-1], np.int32), np.zeros((M, 1), np.int32), u, T, 0,
                                  lib=lib)
    assert (r["path_len"] == 0).all()
    counts = np.bincount(r["out_tokens"][:, 0], minlength=V)
    p = _softmax64(row, T)
    assert np.all(np.abs(counts / M - p) <= 1.0 / M + 1e-6), (counts / M, p)


def check_walk_brute_force(lib, seed=31, T=0.8):
    rng = np.random.default_rng(seed)
    B, V = 40, 9
    for trial in range(6):
        N = int(rng.integers(1, 20))
        parents = tpins._random_tree(rng, N)
        target = (rng.standard_normal((B, N, V)) * 1.5).astype(np.float32)
        u = rng.random((B, N)).astype(np.float32)
        draws = np.zeros((B, N), np.int64)
        margin = np.zeros((B, N))
        for b in range(B):
            for n in range(N):
                draws[b, n], margin[b, n] = _draw(target[b, n], T, u[b, n])
        children = [[c for c in range(N) if parents[c] == n] for n in range(N)]
        tokens = np.zeros((B, N), np.int32)
        for b in range(B):
            for n in range(N):
                pool = list(rng.permutation(V))
                if children[n] and rng.random() < 0.75:  # one child carries the parent's draw
                    pool.remove(draws[b, n])
                    pool.insert(int(rng.integers(0, len(children[n]))), draws[b, n])
                for c, t in zip(children[n], pool):
                    tokens[b, c] = t
        max_depth = int(rng.integers(0, 6))
        r = oracle.verify_tree_sample(target, parents, tokens, u, T, max_depth, lib=lib)
        for b in range(B):
            if margin[b].min() < 1e-9:  # a uniform on a boundary: rounding decides it
                continue
            # the longest root path whose every node carries its parent's draw
            best = [0]
            stack = [[0]]
            while stack:
                path = stack.pop()
                if len(path) - 1 > len(best) - 1:
                    best = path
                if len(path) - 1 < max_depth:
                    for c in children[path[-1]]:
                        if tokens[b, c] == draws[b, path[-1]]:
                            stack.append(path + [c])
            L = len(best) - 1
            assert r["path_len"][b] == L
            assert list(r["path_nodes"][b, :L + 1]) == best
            assert list(r["out_tokens"][b, :L]) == [tokens[b, n] for n in best[1:]]
            assert r["out_tokens"][b, L] == draws[b, best[-1]]
            assert (r["out_tokens"][b, L + 1:] == -1).all()


def check_dominant_logit_is_greedy(lib, seed=41):
    rng = np.random.default_rng(seed)
    B, N, V = 30, 14, 12
    parents = tpins._random_tree(rng, N)
    target = rng.standard_normal((B, N, V)).astype(np.float32)
    spike = rng.integers(0, V, (B, N))
    np.put_along_axis(target, spike[..., None], 80.0, axis=-1)
    tokens = np.where(rng.random((B, N)) < 0.6, spike, rng.integers(0, V, (B, N))).astype(np.int32)
    u = rng.random((B, N)).astype(np.float32)
    g = oracle.verify_tree(target, parents, tokens, 5, lib=lib)
    s = oracle.verify_tree_sample(target, parents, tokens, u, 1.0, 5, lib=lib)
    for k in ("path_len", "path_nodes", "out_tokens"):
        np.testing.assert_array_equal(s[k], g[k])


def test_draw_frequencies_follow_softmax(oracle_lib):
    check_draw_frequencies(oracle_lib)


@pytest.mark.parametrize("T", [0.4, 1.7])
def test_draw_frequencies_other_temperatures(oracle_lib, T):
    check_draw_frequencies(oracle_lib, V=4, T=T, M=8000, seed=int(T * 10))


def test_walk_matches_brute_force(oracle_lib):
    check_walk_brute_force(oracle_lib)


def test_dominant_logit_reduces_to_greedy(oracle_lib):
    check_dominant_logit_is_greedy(oracle_lib)


def test_node_cdf_brackets_every_uniform(oracle_lib):
    rng = np.random.default_rng(7)
    B, N, V = 20, 6, 30
    target = rng.standard_normal((B, N, V)).astype(np.float32)
    u = rng.random((B, N)).astype(np.float32)
    r = oracle.verify_tree_sample(target, tpins._random_tree(rng, N), np.zeros((B, N), np.int32), u, 0.9, 3,
                                  lib=oracle_lib)
    lo, hi = r["node_cdf"][..., 0], r["node_cdf"][..., 1]
    assert np.all(lo <= u) and np.all(u < hi)
