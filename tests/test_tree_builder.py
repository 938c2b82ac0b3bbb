"""The library's sparse-tree builder (spec_build_sparse_tree, host code) against
the oracle's, node for node: the post's K=4, top-8, 64-node tree, random
accuracy tables, exact ties, chains, a node count above the full tree's size,
and the argument checks.  It runs on the host, so these tests need no GPU;
tests/test_gpu_parity.py feeds its tree to the mask kernel and the tree walk.
"""
import ctypes

import numpy as np
import pytest

import oracle
import sampling_online_softmax_gb300 as sv
from sampling_online_softmax_gb300 import build as sv_build


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.load_library()


def synthetic(K, S):
    return np.array([[0.6 * 0.8 ** k * 0.5 ** i for i in range(1, S + 1)] for k in range(1, K + 1)])


def same(acc, n):
    got = sv.spec_build_sparse_tree(acc, n)
    want = oracle.build_sparse_tree(acc, n)
    for k in ("parents", "depth", "rank"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    assert got["expected_len"] == want["expected_len"]
    return got


def test_post_tree_node_for_node(lib):
    t = same(synthetic(4, 8), 64)
    assert len(t["parents"]) == 64 and np.bincount(t["depth"]).tolist() == [1, 8, 28, 26, 1]


@pytest.mark.parametrize("K,S,n,seed", [(3, 5, 40, 0), (4, 8, 64, 1), (2, 10, 25, 2), (6, 3, 100, 3), (1, 12, 7, 4)])
def test_random_tables(lib, K, S, n, seed):
    rng = np.random.default_rng(seed)
    same(rng.uniform(0.0, 1.0, size=(K, S)), n)
    # quantised tables: many exact ties within and across depths
    same(np.round(rng.uniform(0.0, 1.0, size=(K, S)) * 4) / 4, n)


def test_full_tree_and_chain(lib):
    t = same(np.full((3, 4), 0.5), 1000)          # 4 + 16 + 64 nodes below the root: all of them
    assert len(t["parents"]) == 85
    t = same(np.array([[0.9], [0.8], [0.1]]), 10)
    assert t["parents"].tolist() == [-1, 0, 1, 2]
    same(np.zeros((2, 3)), 5)                      # every product 0: the order is the tie rule alone
    same(synthetic(4, 8), 1)                       # the root alone


def test_argument_checks(lib):
    acc = synthetic(2, 3)
    for a, n in ((acc, 0), (acc, 16385), (np.full((2, 3), 1.5), 4), (np.full((2, 3), np.nan), 4),
                 (np.full((65, 1), 0.5), 4), (np.full((2, 3), -0.1), 4)):
        with pytest.raises(sv.SpecError):
            sv.spec_build_sparse_tree(a, n)
    P = ctypes.c_void_p
    buf = np.zeros(8, np.int32)
    nb = ctypes.c_int(0)
    assert lib.spec_build_sparse_tree(None, 2, 3, 4, P(buf.ctypes.data), P(buf.ctypes.data), P(buf.ctypes.data),
                                      ctypes.byref(nb), None) == sv.SPEC_ERR_INVALID_ARG
