"""The benchmark's extra configurations build their inputs on the CPU too: every
generator path ends (no search that cannot finish), with the shapes the GPU
calls expect.  The large configurations are left to the GPU runs."""
import os

import numpy as np
import pytest
import torch

import bench
import oracle


@pytest.mark.parametrize("name", ["small_T1", "small_greedy", "medusa_tree_greedy", "medusa_tree_sampled_T1",
                                  "medusa_tree_mask"])
def test_config_inputs_build_on_cpu(name):
    w, T, kind, d = bench.config_inputs(name, torch.device("cpu"))
    assert kind == bench.CONFIGS[name][2] and T == bench.CONFIGS[name][1]
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


def test_every_config_name_has_a_kind_and_a_kernel():
    kinds = set(k for _, _, k in bench.CONFIGS.values())
    assert kinds <= set(bench.CONFIG_KERNELS)
    assert set(bench.CONFIG_PROFILES) <= set(bench.CONFIGS)


def test_every_profile_the_bench_reads_exists_and_parses():
    # the per-launch traffic comes from these summaries; each names the source hash it was taken on
    import re
    for name in [bench.HEADLINE_PROFILE, *bench.CONFIG_PROFILES.values()]:
        text = open(os.path.join(bench.PROFILES, name)).read()
        h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{16})", text)
        t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
        assert h and t and int(t.group(1)) > 0, name
        assert bench.committed_traffic(name, h.group(1)) == int(t.group(1))
        assert bench.committed_traffic(name, "0" * 16) is None   # another source: no traffic claimed


def test_clock_summary_reads_nvidia_smi_lines():
    lines = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2055, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1250.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    s = bench.summarize_clocks(lines)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.summarize_clocks([])["samples"] == 0


def test_small_config_parity_counts_on_the_cpu():
    """The per-config parity leg: the oracle's own outputs compared with themselves are exact."""
    w, T, kind, d = bench.config_inputs("small_T1", torch.device("cpu"))
    h = {k: bench.to_oracle(v) for k, v in d.items() if hasattr(v, "detach")}
    o = bench.oracle_call(kind, T, h, d)()
    g = {k: o[k] for k in ("accept_len", "out_tokens", "num_emitted")}
    p = bench.config_parity(kind, T, h, o, g)
    assert p["exact"] == w.B and p["failures"] == 0


def test_source_hash_covers_every_kernel_source():
    import os
    h1 = bench.kernel_source_hash()
    assert len(h1) == 16 and int(h1, 16) >= 0
    csrc = os.path.join(bench.ROOT, "sampling_online_softmax_gb300", "csrc")
    assert any(f.startswith("kern_") for f in os.listdir(csrc))
