"""The benchmark's extra configurations build their inputs on the CPU too: every
generator path ends (no search that cannot finish), with the shapes the GPU
calls expect.  The large configurations are left to the GPU runs."""
import numpy as np
import pytest
import torch

import bench
import oracle


@pytest.mark.parametrize("name", ["small", "small_greedy", "medusa_tree", "medusa_tree_sample", "medusa_tree_mask"])
def test_extra_inputs_build_on_cpu(name):
    w, T, kind, d = bench._extra_inputs(name, torch.device("cpu"))
    assert kind == bench.EXTRA[name][2] and T == bench.EXTRA[name][1]
    if kind == "linear":
        assert tuple(d["target"].shape) == (w.B, w.K + 1, w.V)
    elif kind == "mask":
        par = d["parents"].numpy()
        assert par[0] == -1 and all(0 <= par[c] < c for c in range(1, len(par)))
    else:
        B, N = d["node_tokens"].shape
        assert tuple(d["target"].shape) == (B, N, w.V)
        if kind == "tree_sample":
            assert tuple(d["u_nodes"].shape) == (B, N)
            # the walks can go below the root: the oracle accepts at least one node somewhere
            o = oracle.verify_tree_sample(d["target"].numpy(), d["parents"].numpy(), d["node_tokens"].numpy(),
                                          d["u_nodes"].numpy(), T, int(d["max_depth"]))
            assert o["path_len"].max() >= 1


def test_every_extra_name_has_a_kind():
    assert set(k for _, _, k in bench.EXTRA.values()) <= {"linear", "tree", "tree_sample", "rows", "mask"}
