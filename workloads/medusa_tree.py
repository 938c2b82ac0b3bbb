"""Medusa candidate trees, given as parent-index arrays.

"Speculative-Decoding / Medusa" blog:
  section 三 (Attention Tree): head k proposes its top-s_k tokens; the full
    candidate tree is their Cartesian product, with prod_{i<=K} s_i paths and
    sum_{i<=K} prod_{j<=i} s_j nodes (4096 paths and 4680 nodes for K = 4,
    top-8);
  section 四 (optimized tree construction): with a_k^(i) the accuracy of the
    i-th top prediction of head k, assumed independent, the path [i_1..i_m]
    is accepted with probability prod_j a_j^(i_j); the expected accepted
    length is E[L] = sum over the tree's nodes of that product; the tree is
    grown greedily by adding, one node at a time, the candidate whose
    contribution is largest, up to a fixed node count (64 nodes in the post).

Reading for ties (the post is silent): equal contributions are ordered by
smaller depth, then by the lexicographically smaller rank path.  Node 0 is the
root (the last accepted token); nodes are numbered by (depth, rank path), so
every parent index is smaller than its children's.
"""
from __future__ import annotations

import dataclasses
import heapq
import itertools


def synthetic_accuracy(k: int, i: int) -> float:
    """a_k^(i) = 0.6 * 0.8^k * 0.5^i for head k >= 1 and rank i >= 1."""
    return 0.6 * (0.8 ** k) * (0.5 ** i)


@dataclasses.dataclass
class Tree:
    parents: list          # parents[0] = -1
    depth: list            # depth[0] = 0
    rank: list             # rank of the node among its parent's candidates (1-based); 0 for root
    paths: list            # rank path of each node; () for root

    def children(self):
        ch = [[] for _ in self.parents]
        for c, p in enumerate(self.parents):
            if p >= 0:
                ch[p].append(c)
        return ch

    @property
    def n_nodes(self) -> int:
        return len(self.parents)

    def n_paths(self) -> int:
        """Root-to-leaf paths."""
        ch = self.children()
        return sum(1 for c in range(len(self.parents)) if not ch[c] and c != 0) or 1


def _from_paths(paths) -> Tree:
    paths = sorted(set(paths), key=lambda p: (len(p), p))
    index = {p: n for n, p in enumerate(paths)}
    parents, depth, rank = [], [], []
    for p in paths:
        parents.append(-1 if len(p) == 0 else index[p[:-1]])
        depth.append(len(p))
        rank.append(p[-1] if p else 0)
    return Tree(parents, depth, rank, paths)


def path_value(path, acc) -> float:
    """prod_j a_j^(i_j) along a rank path (section 四)."""
    v = 1.0
    for j, i in enumerate(path, start=1):
        v *= acc(j, i)
    return v


def expected_accept_length(tree: Tree, acc) -> float:
    """E[L] = sum over non-root nodes of the product of accuracies along their path."""
    return sum(path_value(p, acc) for p in tree.paths if len(p) > 0)


def cartesian_tree(sizes) -> Tree:
    """Full candidate tree: head k contributes its top-sizes[k-1] tokens at depth k."""
    paths = [()]
    for d in range(1, len(sizes) + 1):
        paths += list(itertools.product(*[range(1, s + 1) for s in sizes[:d]]))
    return _from_paths(paths)


def build_sparse_tree(K: int, s: int, n_nodes: int, acc) -> Tree:
    """Greedy tree of n_nodes nodes (root included) over K heads with top-s candidates."""
    chosen = [()]
    heap = []

    def push(path):
        # max value first; then smaller depth; then lexicographically smaller path
        heapq.heappush(heap, (-path_value(path, acc), len(path), path))

    for i in range(1, s + 1):
        push((i,))
    while len(chosen) < n_nodes and heap:
        _, _, path = heapq.heappop(heap)
        chosen.append(path)
        if len(path) < K:
            for i in range(1, s + 1):
                push(path + (i,))
    return _from_paths(chosen)
