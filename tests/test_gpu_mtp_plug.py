"""spec_mtp_plug on the GPU against the oracle, bit for bit.

The plug-in consumes spec_verify_linear's device outputs directly (no host
round trip in between): at the MTP workload's full size (B=256, K=1,
V=129280, bf16) after a greedy and a T=1 verify, and on small cases that
cover rows longer than a warp (K=40), writing in place, lengths left alone,
and counts outside [0, K+1].
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from workloads import make_linear

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("sampling_online_softmax_gb300")
BAD_LENGTH = 32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()
    torch.cuda.set_device(0)
    oracle.load()


def to_oracle(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_plug_after_verify_at_the_mtp_workload(T):
    d = make_linear(3, T, device="cuda")
    B, K = d["draft_tokens"].shape
    g = torch.Generator(device="cuda").manual_seed(31)
    start = torch.randint(0, 129280, (B, 1), generator=g, device="cuda", dtype=torch.int32)
    inp = torch.cat([start, d["draft_tokens"]], dim=1).contiguous()      # the 2 * B tokens the target scored
    lens = torch.randint(1, 4000, (B,), generator=g, device="cuda", dtype=torch.int32)
    lens0 = lens.clone()
    r = sv.spec_verify_linear(d["target"], d["draft"] if T > 0 else None, d["draft_tokens"], d["u_accept"],
                              d["u_bonus"], T)
    p = sv.spec_mtp_plug(inp, r["out_tokens"], r["num_emitted"], pad=0, seq_lens=lens, status=r["status"])
    torch.cuda.synchronize()
    assert int(r["status"][0]) == 0
    o = oracle.mtp_plug(to_oracle(inp), to_oracle(r["out_tokens"]), to_oracle(r["num_emitted"]), pad=0,
                        seq_lens=to_oracle(lens0))
    np.testing.assert_array_equal(p["next_tokens"].cpu().numpy(), o["next_tokens"])
    np.testing.assert_array_equal(lens.cpu().numpy(), o["seq_lens"])
    # chained with the oracle's own verify: equal wherever the two verifies agree (all but near ties)
    ov = oracle.verify_linear(to_oracle(d["target"]), to_oracle(d["draft"]) if T > 0 else None,
                              to_oracle(d["draft_tokens"]), to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T)
    rep = compare.compare_linear({k: v.cpu().numpy() for k, v in r.items()}, ov, to_oracle(d["u_accept"]),
                                 to_oracle(d["u_bonus"]), T, check_probs=False)
    assert rep.ok
    oc = oracle.mtp_plug(to_oracle(inp), ov["out_tokens"], ov["num_emitted"], pad=0)
    same = np.all(r["out_tokens"].cpu().numpy() == ov["out_tokens"], axis=1)
    np.testing.assert_array_equal(p["next_tokens"].cpu().numpy()[same], oc["next_tokens"][same])
    assert same.sum() >= B - (rep.accept_ties + rep.bonus_ties)


@pytest.mark.parametrize("B,K,in_place,with_lens", [(37, 40, True, True), (37, 40, False, False),
                                                    (9, 0, True, True), (300, 3, True, False)])
def test_plug_edge_cases(B, K, in_place, with_lens):
    rng = np.random.default_rng(B * 100 + K)
    W = K + 1
    inp = rng.integers(0, 1 << 20, (B, W)).astype(np.int32)
    ot = rng.integers(0, 1 << 20, (B, W)).astype(np.int32)
    ne = rng.integers(0, W + 1, B).astype(np.int32)
    ne[: min(B, 3)] = [0, W, 1][: min(B, 3)]
    lens = rng.integers(0, 100, B).astype(np.int32)
    t_in, t_ot, t_ne = (torch.from_numpy(a).cuda() for a in (inp, ot, ne))
    t_lens = torch.from_numpy(lens).cuda() if with_lens else None
    p = sv.spec_mtp_plug(t_in, t_ot, t_ne, pad=-3, seq_lens=t_lens, in_place=in_place)
    torch.cuda.synchronize()
    o = oracle.mtp_plug(inp, ot, ne, pad=-3, seq_lens=lens if with_lens else None)
    np.testing.assert_array_equal(p["next_tokens"].cpu().numpy(), o["next_tokens"])
    if in_place:
        assert p["next_tokens"].data_ptr() == t_in.data_ptr()
    if with_lens:
        np.testing.assert_array_equal(t_lens.cpu().numpy(), o["seq_lens"])
    assert int(p["status"][0]) == 0


def test_plug_flags_counts_out_of_range():
    inp = np.arange(20, dtype=np.int32).reshape(5, 4)
    ot = (100 + np.arange(20, dtype=np.int32)).reshape(5, 4)
    ne = np.array([-1, 5, 4, 0, 2], np.int32)
    lens = np.full(5, 10, np.int32)
    t_lens = torch.from_numpy(lens.copy()).cuda()
    p = sv.spec_mtp_plug(torch.from_numpy(inp).cuda(), torch.from_numpy(ot).cuda(), torch.from_numpy(ne).cuda(),
                         pad=7, seq_lens=t_lens)
    torch.cuda.synchronize()
    o = oracle.mtp_plug(inp, ot, ne, pad=7, seq_lens=lens)
    assert o["bad"] and int(p["status"][0]) == BAD_LENGTH
    np.testing.assert_array_equal(p["next_tokens"].cpu().numpy(), o["next_tokens"])
    np.testing.assert_array_equal(t_lens.cpu().numpy(), o["seq_lens"])
