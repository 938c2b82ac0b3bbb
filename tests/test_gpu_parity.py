"""GPU library vs the CPU oracle, element by element, through the C ABI.

Every workload runs at its full size in the same call the benchmark times,
and small cases cover the edges: K = 0, V = 1, vocabularies smaller than one
16-byte group per CTA, ragged V (rows not 16-byte aligned), K > 32, tiny and
large temperatures, exact ties in greedy mode, no extra token, the extra token
alone, trees of several shapes, and the device status bits.

Integers (accepted lengths, tokens, paths) must be equal except at counted
near ties (oracle/compare.py); probabilities within 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from workloads import WORKLOADS, make_linear, make_tree

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("sampling_online_softmax_gb300")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.load_library()
    torch.cuda.set_device(0)
    oracle.load()


def to_oracle(t):
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def run_linear(d, T, probs=True, with_bonus=True, stream=None):
    draft = d["draft"] if T > 0 else None
    ub = d["u_bonus"] if with_bonus else None
    r = sv.spec_verify_linear(d["target"], draft, d["draft_tokens"], d["u_accept"], ub, T, probs=probs and T > 0,
                              stream=stream)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in r.items()}
    o = oracle.verify_linear(to_oracle(d["target"]), to_oracle(draft), to_oracle(d["draft_tokens"]),
                             to_oracle(d["u_accept"]), to_oracle(ub), T)
    return g, o


def assert_parity(g, o, d, T, with_bonus=True, status_ok=True, check_probs=True):
    rep = compare.compare_linear(g, o, to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]) if with_bonus else None, T,
                                 check_probs=check_probs)
    print(rep.summary())
    assert rep.ok, rep.failures[:8]
    if status_ok:
        assert int(g["status"][0]) == 0, "device status bits %#x" % int(g["status"][0])
    # invariants the pages fix: at most K + 1 tokens, the extra token present
    K = o["out_tokens"].shape[1] - 1
    assert ((g["accept_len"] >= 0) & (g["accept_len"] <= K)).all()
    assert (g["num_emitted"] == g["accept_len"] + (1 if with_bonus else 0)).all()
    return rep


# ------------------------------------------------------------ full workloads

@pytest.mark.parametrize("number,T", [(1, 1.0), (1, 0.0), (2, 0.7), (3, 0.0), (3, 1.0), (5, 0.7)])
def test_workload_parity_full_size(number, T):
    d = make_linear(number, T, device="cuda")
    g, o = run_linear(d, T)
    rep = assert_parity(g, o, d, T)
    # near ties are rare: a handful per thousand sequences at most
    assert rep.accept_ties + rep.bonus_ties <= max(2, rep.sequences // 50)


def test_medusa_tree_workload_full_size():
    d = make_tree(4, device="cuda")
    r = sv.spec_verify_tree(d["target"], d["parents"], d["node_tokens"], d["max_depth"])
    torch.cuda.synchronize()
    o = oracle.verify_tree(to_oracle(d["target"]), to_oracle(d["parents"]), to_oracle(d["node_tokens"]),
                           d["max_depth"])
    rep = compare.compare_tree({k: v.cpu().numpy() for k, v in r.items()}, o)
    assert rep.ok, rep.failures[:5]
    assert int(r["status"][0]) == 0
    assert o["path_len"].max() >= 1       # the workload does accept candidates


# ---------------------------------------------------------------- edge cases

def rand_linear(B, K, V, dtype, seed, scale=2.0, noise=0.8, quant=None, T=1.0):
    g = torch.Generator().manual_seed(seed)
    t = scale * torch.randn((B, K + 1, V), generator=g)
    if quant:
        t = torch.round(t * quant) / quant
    d = t[:, :K] + noise * torch.randn((B, K, V), generator=g)
    if K > 0:
        am = torch.argmax(t[:, :K], dim=-1)
        rnd = torch.randint(0, V, (B, K), generator=g)
        tokens = torch.where(torch.rand((B, K), generator=g) < 0.6, am, rnd).to(torch.int32)
    else:
        tokens = torch.zeros((B, 0), dtype=torch.int32)
    u = torch.rand((B, K), generator=g)
    ub = torch.rand((B,), generator=g)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    return dict(target=t.to(dt).cuda(), draft=d.to(dt).cuda(), draft_tokens=tokens.cuda(), u_accept=u.cuda(),
                u_bonus=ub.cuda())


EDGE = [
    # B, K, V, dtype, T
    (3, 0, 1000, "f32", 1.0),       # no draft: one token from p_0
    (3, 2, 1, "bf16", 0.8),         # one-token vocabulary
    (5, 3, 7, "f32", 1.0),          # fewer elements than CTAs
    (4, 3, 29, "bf16", 0.5),
    (4, 40, 300, "bf16", 1.2),      # K > 32: more than one ballot
    (7, 3, 5003, "bf16", 0.7),      # ragged rows (V * 2 % 16 != 0)
    (7, 3, 4099, "f32", 0.9),       # ragged rows, fp32
    (6, 2, 50000, "f32", 1e-3),     # near-greedy temperature
    (6, 2, 20000, "bf16", 100.0),   # nearly flat distributions
    (2, 2, 262147, "bf16", 1.0),    # large, ragged vocabulary
    (9, 5, 32000, "f32", 0.0),      # greedy
    (9, 4, 5003, "bf16", 0.0),      # greedy, ragged
]


@pytest.mark.parametrize("B,K,V,dtype,T", EDGE)
def test_linear_edge_cases(B, K, V, dtype, T):
    d = rand_linear(B, K, V, dtype, seed=B * 1000 + K * 10 + V % 97)
    g, o = run_linear(d, T)
    assert_parity(g, o, d, T)


def test_greedy_exact_ties_take_lowest_index():
    d = rand_linear(16, 4, 3001, "bf16", seed=5, quant=1.0)   # integer logits: many ties at the max
    g, o = run_linear(d, 0.0)
    assert_parity(g, o, d, 0.0)


def test_extreme_uniforms_for_the_extra_token():
    # u_b at the ends of [0, 1): zero, the smallest subnormal, a subnormal, a tiny normal, one half and
    # the largest float below one; the draw takes the first / last positive weight at the ends
    us = np.array([0.0, 1.4e-45, 1e-40, 1e-30, 0.5, np.nextafter(np.float32(1), np.float32(0))], dtype=np.float32)
    for dtype, T in (("bf16", 0.7), ("f32", 1.0)):
        d = rand_linear(len(us), 3, 5003, dtype, seed=17)
        d["u_bonus"] = torch.from_numpy(us).cuda()
        g, o = run_linear(d, T)
        assert_parity(g, o, d, T)


def test_no_extra_token_and_no_probs():
    d = rand_linear(8, 3, 7001, "bf16", seed=6)
    g, o = run_linear(d, 0.9, probs=False, with_bonus=False)
    assert_parity(g, o, d, 0.9, with_bonus=False, check_probs=False)
    assert (g["num_emitted"] == g["accept_len"]).all()


def test_non_default_stream_and_repeat_calls_are_identical():
    d = make_linear(2, 0.7, device="cuda", B=16)
    s = torch.cuda.Stream()
    g1, o = run_linear(d, 0.7, stream=s)
    g2, _ = run_linear(d, 0.7, stream=s)
    for k in ("accept_len", "out_tokens", "num_emitted", "probs"):
        np.testing.assert_array_equal(g1[k], g2[k])
    assert_parity(g1, o, d, 0.7)


def test_workspace_left_zeroed():
    d = rand_linear(5, 3, 3000, "f32", seed=7)
    ws = torch.zeros(sv.spec_workspace_bytes_linear(5, 3, 3000, torch.float32), dtype=torch.uint8, device="cuda")
    sv.spec_verify_linear(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"], 1.0,
                          workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.sum()) == 0              # counters and per-unit entries all reset


def test_one_workspace_shared_by_different_shapes():
    """A workspace used by a (B=3, K=2) call then serves a (B=6, K=3) call and a tree call."""
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    for B, K, V, T, seed in ((3, 2, 999, 1.0, 21), (6, 3, 1001, 0.8, 22), (6, 3, 1001, 0.0, 23), (2, 7, 500, 1.0, 24)):
        d = rand_linear(B, K, V, "f32", seed=seed)
        r = sv.spec_verify_linear(d["target"], d["draft"] if T > 0 else None, d["draft_tokens"], d["u_accept"],
                                  d["u_bonus"], T, probs=T > 0, workspace=ws)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in r.items()}
        o = oracle.verify_linear(to_oracle(d["target"]), to_oracle(d["draft"]) if T > 0 else None,
                                 to_oracle(d["draft_tokens"]), to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T)
        assert_parity(g, o, d, T)
        assert int(ws.sum()) == 0
    t, par, tok = _random_tree_inputs(5, 9, 300, "f32", seed=3)
    r = sv.spec_verify_tree(t, par, tok, 4, workspace=ws)
    torch.cuda.synchronize()
    o = oracle.verify_tree(to_oracle(t), to_oracle(par), to_oracle(tok), 4)
    assert compare.compare_tree({k: v.cpu().numpy() for k, v in r.items()}, o).ok
    assert int(ws.sum()) == 0


# ----------------------------------------------------------- extra token alone

@pytest.mark.parametrize("B,K,V,dtype,T", [(32, 4, 32000, "f32", 1.0), (17, 3, 5003, "bf16", 0.7),
                                           (9, 2, 20000, "bf16", 0.0), (4, 0, 999, "f32", 1.0)])
def test_sample_bonus_parity(B, K, V, dtype, T):
    d = rand_linear(B, K, V, dtype, seed=11 + B)
    al = torch.randint(0, K + 1, (B,), generator=torch.Generator().manual_seed(3)).to(torch.int32)
    draft = d["draft"] if T > 0 else None
    r = sv.spec_sample_bonus(d["target"], draft, al.cuda(), d["u_bonus"], T)
    torch.cuda.synchronize()
    o = oracle.sample_bonus(to_oracle(d["target"]), to_oracle(draft), al.numpy(), to_oracle(d["u_bonus"]), T)
    rep = compare.compare_bonus(r["bonus_token"].cpu().numpy(), o, to_oracle(d["u_bonus"]), T)
    assert rep.ok, rep.failures[:5]
    assert int(r["status"][0]) == 0


def test_sample_bonus_matches_fused_extra_token():
    d = make_linear(2, 0.7, device="cuda", B=24)
    r = sv.spec_verify_linear(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"], 0.7)
    b = sv.spec_sample_bonus(d["target"], d["draft"], r["accept_len"], d["u_bonus"], 0.7)
    torch.cuda.synchronize()
    j = r["accept_len"].long()
    fused = r["out_tokens"].gather(1, j[:, None])[:, 0]
    assert torch.equal(fused, b["bonus_token"])


# -------------------------------------------------------------------- trees

def _random_tree_inputs(B, N, V, dtype, seed):
    rng = np.random.default_rng(seed)
    parents = np.array([-1] + [int(rng.integers(0, c)) for c in range(1, N)], np.int32)
    t = torch.from_numpy(rng.standard_normal((B, N, V)).astype(np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    am = torch.argmax(t.float(), dim=-1).numpy()
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(N):
            ch = [c for c in range(N) if parents[c] == n]
            pool = list(rng.permutation(V)[:len(ch) + 1])
            if am[b, n] in pool:
                pool.remove(am[b, n])
            if ch and rng.random() < 0.75:
                pool.insert(int(rng.integers(0, len(ch))), am[b, n])
            for c, tok in zip(ch, pool):
                tokens[b, c] = tok
    return t.cuda(), torch.from_numpy(parents).cuda(), torch.from_numpy(tokens).cuda()


@pytest.mark.parametrize("B,N,V,dtype,depth", [(8, 1, 1000, "f32", 3), (12, 30, 5003, "bf16", 6),
                                               (6, 100, 2048, "f32", 4), (4, 20, 777, "f32", 0)])
def test_tree_parity(B, N, V, dtype, depth):
    t, par, tok = _random_tree_inputs(B, N, V, dtype, seed=N + V)
    r = sv.spec_verify_tree(t, par, tok, depth)
    torch.cuda.synchronize()
    o = oracle.verify_tree(to_oracle(t), to_oracle(par), to_oracle(tok), depth)
    rep = compare.compare_tree({k: v.cpu().numpy() for k, v in r.items()}, o)
    assert rep.ok, rep.failures[:5]


def test_chain_tree_equals_linear_greedy_on_gpu():
    d = rand_linear(20, 5, 4000, "bf16", seed=12, quant=2.0)
    lin = sv.spec_verify_linear(d["target"], None, d["draft_tokens"], None, d["u_bonus"], 0.0)
    par = torch.arange(-1, 5, dtype=torch.int32, device="cuda")
    nt = torch.cat([torch.zeros((20, 1), dtype=torch.int32, device="cuda"), d["draft_tokens"]], 1).contiguous()
    tr = sv.spec_verify_tree(d["target"], par, nt, 5)
    torch.cuda.synchronize()
    assert torch.equal(tr["path_len"], lin["accept_len"])
    assert torch.equal(tr["out_tokens"], lin["out_tokens"])


# ------------------------------------------------------- sampled trees

def _draws(target, T, u):
    """Each node's draw from softmax(target / T) at uniform u (float64, on the host): used
    only to build node tokens that make the walks long."""
    x = target.float().cpu().double().numpy() / T
    p = np.exp(x - x.max(-1, keepdims=True))
    c = np.cumsum(p, -1)
    want = u.cpu().double().numpy()[..., None] * c[..., -1:]
    return np.minimum((c <= want).sum(-1), x.shape[-1] - 1)


def _sampled_tree_inputs(t, parents, T, seed, hit=0.75):
    B, N, V = t.shape
    rng = np.random.default_rng(seed)
    u = torch.from_numpy(rng.random((B, N)).astype(np.float32)).cuda()
    dr = _draws(t, T, u)
    par = parents.cpu().numpy()
    children = [[c for c in range(N) if par[c] == n] for n in range(N)]
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(N):
            ch = children[n]
            if not ch:
                continue
            pool = [int(v) for v in rng.permutation(V)[:len(ch) + 1] if v != dr[b, n]]
            if rng.random() < hit:
                pool.insert(int(rng.integers(0, len(ch))), int(dr[b, n]))
            for c, tok in zip(ch, pool):
                tokens[b, c] = tok
    return u, torch.from_numpy(tokens).cuda()


def _tree_sample_parity(t, par, tok, u, T, depth):
    r = sv.spec_verify_tree_sample(t, par, tok, u, T, depth)
    torch.cuda.synchronize()
    o = oracle.verify_tree_sample(to_oracle(t), to_oracle(par), to_oracle(tok), to_oracle(u), T, depth)
    rep = compare.compare_tree_sample({k: v.cpu().numpy() for k, v in r.items()}, o, to_oracle(u))
    print(rep.summary())
    assert rep.ok, rep.failures[:5]
    assert int(r["status"].item()) == 0
    return r, o


def test_medusa_tree_workload_sampled_full_size():
    """The Medusa tree workload's shapes (B=16, 64 nodes, V=32000 fp32) with the choice drawn at T = 1."""
    d = make_tree(4, device="cuda")
    u, tok = _sampled_tree_inputs(d["target"], d["parents"], 1.0, seed=404)
    r, o = _tree_sample_parity(d["target"], d["parents"], tok, u, 1.0, d["max_depth"])
    assert o["path_len"].max() >= 2   # the walks go below the root


@pytest.mark.parametrize("B,N,V,dtype,depth,T", [(8, 1, 1000, "f32", 3, 1.0), (12, 30, 5003, "bf16", 6, 0.7),
                                                 (6, 100, 2048, "f32", 4, 1.5), (4, 20, 777, "f32", 0, 0.9),
                                                 (3, 9, 7, "bf16", 5, 2.0)])
def test_tree_sample_parity(B, N, V, dtype, depth, T):
    t, par, _ = _random_tree_inputs(B, N, V, dtype, seed=N + V + 1)
    u, tok = _sampled_tree_inputs(t, par, T, seed=N * V)
    _tree_sample_parity(t, par, tok, u, T, depth)


def test_tree_sample_with_dominant_logits_equals_greedy_walk():
    t, par, tok = _random_tree_inputs(10, 25, 3000, "f32", seed=99)
    am = torch.argmax(t, dim=-1, keepdim=True)
    t = t.scatter(-1, am, 90.0).contiguous()     # every draw is the argmax
    u = torch.rand((10, 25), device="cuda")
    g = sv.spec_verify_tree(t, par, tok, 5)
    s = sv.spec_verify_tree_sample(t, par, tok, u, 1.0, 5)
    torch.cuda.synchronize()
    for k in ("path_len", "path_nodes", "out_tokens"):
        assert torch.equal(g[k], s[k]), k


def test_tree_sample_workspace_left_zeroed_and_repeatable():
    t, par, _ = _random_tree_inputs(5, 12, 4099, "bf16", seed=5)
    u, tok = _sampled_tree_inputs(t, par, 0.8, seed=6)
    nbytes = sv.spec_workspace_bytes_tree_sample(5, 12, 4099, t.dtype)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    a = sv.spec_verify_tree_sample(t, par, tok, u, 0.8, 4, workspace=ws)
    b = sv.spec_verify_tree_sample(t, par, tok, u, 0.8, 4, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0
    for k in ("path_len", "path_nodes", "out_tokens"):
        assert torch.equal(a[k], b[k]), k


# ------------------------------------------------------------- row sampler

@pytest.mark.parametrize("B,V,dtype,T", [(64, 128256, "bf16", 0.7), (64, 128256, "bf16", 0.0), (300, 5003, "bf16", 1.3),
                                         (7, 1, "f32", 1.0), (5, 33, "f32", 0.05), (40, 32000, "f32", 4.0)])
def test_sample_rows_parity(B, V, dtype, T):
    rng = np.random.default_rng(B * 7 + V)
    x = torch.from_numpy((rng.standard_normal((B, V)) * 4.0).astype(np.float32))
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    x = x.cuda()
    u = torch.from_numpy(rng.random(B).astype(np.float32)).cuda()
    r = sv.spec_sample_rows(x, u if T > 0 else None, T)
    torch.cuda.synchronize()
    o = oracle.sample_rows(to_oracle(x), to_oracle(u) if T > 0 else None, T)
    g = r["tokens"].cpu().numpy()
    un = to_oracle(u)
    bad = [b for b in range(B) if g[b] != o["tokens"][b]
           and not (T > 0 and min(abs(un[b] - o["cdf"][b, 0]), abs(un[b] - o["cdf"][b, 1])) < compare.NEAR_TIE)]
    assert not bad, [(b, int(g[b]), int(o["tokens"][b])) for b in bad[:5]]
    assert int(r["status"].item()) == 0


def test_sample_rows_equals_extra_token_at_the_tail():
    """A zero-length draft: the extra token of each sequence is a draw from its one target row."""
    rng = np.random.default_rng(77)
    B, V = 20, 3001
    x = torch.from_numpy(rng.standard_normal((B, V)).astype(np.float32) * 3).cuda()
    u = torch.from_numpy(rng.random(B).astype(np.float32)).cuda()
    rows = sv.spec_sample_rows(x, u, 0.9)
    bonus = sv.spec_sample_bonus(x.view(B, 1, V), None, torch.zeros(B, dtype=torch.int32, device="cuda"), u, 0.9)
    torch.cuda.synchronize()
    assert torch.equal(rows["tokens"], bonus["bonus_token"])


# ------------------------------------------------------- tree attention mask

def _mask_parity(parents_np):
    par = torch.from_numpy(np.ascontiguousarray(parents_np, dtype=np.int32)).cuda()
    r = sv.spec_tree_mask(par)
    torch.cuda.synchronize()
    o = oracle.tree_mask(parents_np)
    np.testing.assert_array_equal(r["mask"].cpu().numpy().view(np.uint32), o["mask"])
    np.testing.assert_array_equal(r["depth"].cpu().numpy(), o["depth"])
    assert (int(r["status"].item()) & 16 != 0) == o["bad"]


@pytest.mark.parametrize("N,seed", [(1, 0), (31, 1), (32, 2), (33, 3), (200, 4), (1000, 5), (4099, 6)])
def test_tree_mask_parity(N, seed):
    rng = np.random.default_rng(seed)
    _mask_parity(np.array([-1] + [int(rng.integers(max(0, c - 6), c)) for c in range(1, N)], np.int32))


def test_tree_mask_of_the_medusa_tree_and_a_chain():
    d = make_tree(4, device="cpu", B=1, V=64)
    _mask_parity(d["parents"].numpy())
    _mask_parity(np.arange(-1, 700, dtype=np.int32))


def test_built_tree_feeds_the_mask_and_the_walk():
    """The library's builder (host) makes the post's 64-node tree; the mask kernel and the greedy
    walk consume its parent array as it is, and both agree with the oracle on the oracle's tree."""
    acc = np.array([[0.6 * 0.8 ** k * 0.5 ** i for i in range(1, 9)] for k in range(1, 5)])
    built = sv.spec_build_sparse_tree(acc, 64)
    ot = oracle.build_sparse_tree(acc, 64)
    np.testing.assert_array_equal(built["parents"], ot["parents"])
    par = torch.from_numpy(built["parents"]).cuda()
    m = sv.spec_tree_mask(par)
    torch.cuda.synchronize()
    o = oracle.tree_mask(ot["parents"])
    assert np.array_equal(m["mask"].cpu().numpy().view(np.uint32), o["mask"])
    np.testing.assert_array_equal(m["depth"].cpu().numpy(), ot["depth"])
    # the greedy walk over the built tree, with node tokens that follow the argmax on a random part of it
    g = torch.Generator().manual_seed(8)
    B, N, V = 12, 64, 3000
    target = 3.0 * torch.randn((B, N, V), generator=g)
    am = target.argmax(-1)
    tok = torch.randint(0, V, (B, N), generator=g, dtype=torch.int32)
    hit = torch.rand((B, N), generator=g) < 0.6
    p_idx = torch.from_numpy(built["parents"]).long().clamp(min=0)
    tok = torch.where(hit, am[:, p_idx].to(torch.int32), tok)
    tok[:, 0] = 0
    D = int(built["depth"].max())
    r = sv.spec_verify_tree(target.cuda(), par, tok.cuda(), D)
    torch.cuda.synchronize()
    ow = oracle.verify_tree(target.numpy(), ot["parents"], tok.numpy(), D)
    rep = compare.compare_tree({k: v.cpu().numpy() for k, v in r.items()}, ow)
    assert rep.ok, rep.failures[:5]
    assert ow["path_len"].max() >= 2


def test_tree_mask_flags_a_bad_parent():
    _mask_parity(np.array([-1, 0, 7, 1, 2, 3], np.int32))


# -------------------------------------------------------------- status bits

def test_bad_token_is_flagged_and_rejected():
    d = rand_linear(4, 3, 1000, "f32", seed=13)
    d["draft_tokens"][1, 0] = 1000
    d["draft_tokens"][2, 1] = -5
    r = sv.spec_verify_linear(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"], 1.0)
    torch.cuda.synchronize()
    assert int(r["status"][0]) & sv.DEV_BAD_TOKEN
    assert int(r["accept_len"][1]) == 0
    assert int(r["accept_len"][2]) <= 1


def test_nonfinite_row_is_flagged():
    d = rand_linear(3, 2, 2000, "f32", seed=14)
    d["target"][1, 1, 77] = float("nan")
    r = sv.spec_verify_linear(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"], 1.0)
    torch.cuda.synchronize()
    assert int(r["status"][0]) & sv.DEV_NONFINITE


def test_bad_accept_len_and_bad_tree_are_flagged():
    d = rand_linear(3, 2, 2000, "bf16", seed=15)
    al = torch.tensor([0, 5, -1], dtype=torch.int32, device="cuda")
    r = sv.spec_sample_bonus(d["target"], d["draft"], al, d["u_bonus"], 1.0)
    torch.cuda.synchronize()
    assert int(r["status"][0]) & sv.DEV_BAD_LENGTH
    assert r["bonus_token"][1].item() == -1 and r["bonus_token"][2].item() == -1
    assert r["bonus_token"][0].item() >= 0
    t, par, tok = _random_tree_inputs(2, 6, 100, "f32", seed=1)
    par[3] = 4                                            # not topological
    rt = sv.spec_verify_tree(t, par, tok, 3)
    torch.cuda.synchronize()
    assert int(rt["status"][0]) & sv.DEV_BAD_TREE
