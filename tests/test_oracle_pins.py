"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself or with the GPU path.  Each test
checks a fact that holds independently of how the oracle is written:

  * at most K + 1 tokens per step, the extra token always present, accepted
    tokens are the draft's ("Beschleunigung von Sonar durch Spekulation",
    section "Spekulatives Decoding");
  * speculative sampling leaves the target distribution unchanged -- checked
    exactly by enumerating every draft sequence on a tiny vocabulary, with
    prefix-dependent target and draft models (the property of the method the
    page cites in section "Ziel-Entwurf");
  * greedy mode equals plain argmax decoding (numpy's argmax, lowest index);
  * closed forms: hand-worked three-token example, the probability of a spiked
    token in a constant row, temperature -> 0 reducing to greedy;
  * the residual never re-emits the rejected draft token;
  * bf16 decoding equals fp32 input with the same values.

The functions take the oracle library as an argument so that
test_oracle_mutants.py can run them against deliberately broken builds.
"""
import itertools

import numpy as np
import pytest

import oracle


# ---------------------------------------------------------------- helpers

def softmax64(logits_f32, T):
    z = np.asarray(logits_f32, np.float64) / T
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def next_f32_at_least(x):
    """Smallest float32 >= x (x a float64 in [0, 1])."""
    f = np.float32(x)
    if float(f) < x:
        f = np.nextafter(f, np.float32(2.0))
    return f


def next_f32_above(x):
    """Smallest float32 > x."""
    f = np.float32(x)
    if float(f) <= x:
        f = np.nextafter(f, np.float32(2.0))
    return f


def largest_f32_below(x):
    f = np.float32(x)
    if float(f) >= x:
        f = np.nextafter(f, np.float32(-1.0))
    return f


# ------------------------------------------- exact distribution preservation

def _tables(V, K, seed, scale):
    """Prefix-dependent target and draft 'models': a logits row per prefix."""
    rng = np.random.default_rng(seed)
    T_tab, D_tab = {}, {}
    for m in range(K + 1):
        for pre in itertools.product(range(V), repeat=m):
            T_tab[pre] = (scale * rng.standard_normal(V)).astype(np.float32)
            if m < K:
                D_tab[pre] = (scale * rng.standard_normal(V)).astype(np.float32)
    return T_tab, D_tab


def exact_output_distribution(lib, V, K, T, seed, scale=1.5):
    """Enumerate all V^K drafts; return (joint outcome probabilities, tables).

    Outcome = tuple of emitted tokens (accepted draft tokens + extra token).
    The acceptance probability of position i is the threshold the oracle
    reports, whose use in the decision is probed at the adjacent float32
    uniforms; the extra token's distribution is read from the oracle's
    inverse-CDF intervals by walking u_b across [0, 1)."""
    T = float(np.float32(T))          # the oracle receives T as a float32
    T_tab, D_tab = _tables(V, K, seed, scale)
    xs = list(itertools.product(range(V), repeat=K))
    B = len(xs)
    target = np.stack([np.stack([T_tab[x[:i]] for i in range(K + 1)]) for x in xs])
    draft = np.stack([np.stack([D_tab[x[:i]] for i in range(K)]) for x in xs]) \
        if K > 0 else np.zeros((B, 0, V), np.float32)
    tokens = np.array(xs, np.int32).reshape(B, K)
    Q = np.array([np.prod([softmax64(D_tab[x[:i]], T)[x[i]] for i in range(K)]) for x in xs])

    zeros = np.zeros((B, K), np.float32)
    r = oracle.verify_linear(target, draft, tokens, zeros, None, T, lib=lib)
    thr = r["probs"][:, :, 2]
    assert (r["accept_len"] == K).all()   # u = 0 accepts whenever p(x) > 0

    # the decision switches exactly at the reported threshold (float32 resolution)
    for i in range(K):
        for side in ("below", "at"):
            u = np.zeros((B, K), np.float32)
            live = (thr[:, i] > 0) & (thr[:, i] < 1)
            for b in np.nonzero(live)[0]:
                u[b, i] = largest_f32_below(thr[b, i]) if side == "below" else next_f32_at_least(thr[b, i])
            rr = oracle.verify_linear(target, draft, tokens, u, None, T, lib=lib)
            al = rr["accept_len"][live]
            if side == "below":
                assert (al > i).all(), "accepted below the threshold must hold"
            else:
                assert (al == i).all(), "rejection at the threshold must hold"

    # extra-token intervals for each rejection point j (and the tail j == K)
    masses = {}   # (b, j) -> {token: mass}
    for j in range(K + 1):
        al = np.full(B, j, np.int32)
        u = np.zeros(B, np.float32)
        prev_hi = np.zeros(B)
        done = np.zeros(B, bool)
        for b in range(B):
            masses[(b, j)] = {}
        for _ in range(4 * V + 4):
            rb = oracle.sample_bonus(target, draft, al, u, T, lib=lib)
            lo, hi = rb["bonus_cdf"][:, 0], rb["bonus_cdf"][:, 1]
            for b in np.nonzero(~done)[0]:
                assert lo[b] == prev_hi[b], "inverse-CDF intervals must tile [0, 1)"
                tok = int(rb["bonus_token"][b])
                masses[(b, j)][tok] = masses[(b, j)].get(tok, 0.0) + (hi[b] - lo[b])
                prev_hi[b] = hi[b]
                if hi[b] >= 1.0:
                    done[b] = True
                else:
                    u[b] = next_f32_above(hi[b])
            if done.all():
                break
        assert done.all()

    joint = {}
    for b, x in enumerate(xs):
        acc = 1.0
        for j in range(K + 1):
            pj = acc * ((1.0 - thr[b, j]) if j < K else 1.0)
            if pj > 0:
                for tok, mass in masses[(b, j)].items():
                    y = tuple(x[:j]) + (tok,)
                    joint[y] = joint.get(y, 0.0) + Q[b] * pj * mass
            if j < K:
                acc *= thr[b, j]
    return joint, T_tab


@pytest.mark.parametrize("V,K,T,seed", [
    (3, 1, 1.0, 1), (4, 2, 1.0, 2), (5, 2, 0.7, 3), (3, 3, 1.3, 4), (8, 1, 0.8, 5), (4, 3, 0.5, 6),
])
def test_rejection_sampling_preserves_target_distribution(oracle_lib, V, K, T, seed):
    check_distribution_preserved(oracle_lib, V, K, T, seed)


def check_distribution_preserved(lib, V, K, T, seed):
    joint, T_tab = exact_output_distribution(lib, V, K, T, seed)
    T = float(np.float32(T))
    total = sum(joint.values())
    assert abs(total - 1.0) < 1e-12
    # every emitted token, given the tokens before it, follows the target's
    # distribution at that prefix
    for m in range(K + 1):
        marg = {}
        for y, pr in joint.items():
            if len(y) >= m + 1:
                marg[y[:m + 1]] = marg.get(y[:m + 1], 0.0) + pr
        pre_mass = {}
        for y, pr in marg.items():
            pre_mass[y[:m]] = pre_mass.get(y[:m], 0.0) + pr
        for pre, pm in pre_mass.items():
            p = softmax64(T_tab[pre], T)
            for v in range(V):
                got = marg.get(pre + (v,), 0.0)
                assert abs(got - pm * p[v]) < 1e-12, (m, pre, v, got, pm * p[v])
    # the first token is distributed exactly as p_0
    p0 = softmax64(T_tab[()], T)
    first = np.zeros(V)
    for y, pr in joint.items():
        first[y[0]] += pr
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)


# ------------------------------------------------------------ closed forms

def test_hand_worked_three_token_example(oracle_lib):
    """p = (0.5, 0.3, 0.2), q = (0.2, 0.3, 0.5) at T = 1; tail p_1 = (0.1, 0.6, 0.3).

    x = 0: p/q = 2.5 -> always accepted;  x = 1: ratio 1 -> always accepted;
    x = 2: ratio 0.4 -> accepted iff u < 0.4, else the residual max(0, p - q) =
    (0.3, 0, 0) always gives token 0.  After an acceptance the extra token
    comes from p_1: u_b = 0.05 -> 0, 0.65 -> 1, 0.71 -> 2."""
    t_row0 = np.log([0.5, 0.3, 0.2]).astype(np.float32)
    t_row1 = np.log([0.1, 0.6, 0.3]).astype(np.float32)
    d_row0 = np.log([0.2, 0.3, 0.5]).astype(np.float32)
    cases = [  # x, u, u_b, expected accept_len, expected extra token
        (0, 0.999, 0.05, 1, 0), (0, 0.5, 0.65, 1, 1), (1, 0.9, 0.71, 1, 2),
        (2, 0.39, 0.65, 1, 1), (2, 0.41, 0.99, 0, 0), (2, 0.95, 0.0, 0, 0),
    ]
    B = len(cases)
    target = np.stack([np.stack([t_row0, t_row1])] * B)
    draft = np.stack([d_row0[None]] * B)
    tokens = np.array([[c[0]] for c in cases], np.int32)
    u = np.array([[c[1]] for c in cases], np.float32)
    ub = np.array([c[2] for c in cases], np.float32)
    r = oracle.verify_linear(target, draft, tokens, u, ub, 1.0, lib=oracle_lib)
    for b, (x, _, _, j, tok) in enumerate(cases):
        assert r["accept_len"][b] == j
        assert r["num_emitted"][b] == j + 1
        assert r["out_tokens"][b, j] == tok
        if j == 1:
            assert r["out_tokens"][b, 0] == x
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.3, 0.5])
    for b, (x, *_rest) in enumerate(cases):
        assert abs(r["probs"][b, 0, 0] - p[x]) < 1e-6
        assert abs(r["probs"][b, 0, 1] - q[x]) < 1e-6
        assert abs(r["probs"][b, 0, 2] - min(1.0, p[x] / q[x])) < 1e-6


@pytest.mark.parametrize("V,a,T", [(1000, 5.0, 1.0), (32000, 20.0, 0.7), (7, -3.0, 2.0)])
def test_spiked_constant_row_closed_form(oracle_lib, V, a, T):
    """Row of zeros with one logit a at token s: p(s) = e^{a/T} / (e^{a/T} + V - 1)."""
    s = V // 3
    T = float(np.float32(T))          # the oracle receives T as a float32
    row = np.zeros(V, np.float32)
    row[s] = a
    other = (s + 1) % V
    target = np.stack([row, row])[None]
    draft = np.zeros((1, 1, V), np.float32)
    for x, expect in ((s, np.exp(a / T) / (np.exp(a / T) + V - 1)),
                      (other, 1.0 / (np.exp(a / T) + V - 1))):
        r = oracle.verify_linear(target, draft, np.array([[x]], np.int32),
                                 np.zeros((1, 1), np.float32), None, T, lib=oracle_lib)
        # sequential double summation of V terms: error at most about V * eps
        assert abs(r["probs"][0, 0, 0] - expect) <= 2.0 * V * np.finfo(np.float64).eps * max(1e-300, expect) + 1e-300
        assert abs(r["probs"][0, 0, 1] - 1.0 / V) <= 1e-15


def test_greedy_equals_argmax_decoding(oracle_lib):
    rng = np.random.default_rng(11)
    B, K, V = 40, 5, 257
    # coarse values force exact ties; argmax must take the lowest index
    target = rng.integers(-4, 5, size=(B, K + 1, V)).astype(np.float32)
    am = target.argmax(axis=-1)                       # numpy: first occurrence
    tokens = am[:, :K].copy()
    flip = rng.random((B, K)) < 0.25
    tokens[flip] = (tokens[flip] + 1 + rng.integers(0, V - 1, flip.sum())) % V
    tokens = tokens.astype(np.int32)
    r = oracle.verify_linear(target, None, tokens, None, np.zeros(B, np.float32), 0.0, lib=oracle_lib)
    for b in range(B):
        j = next((i for i in range(K) if tokens[b, i] != am[b, i]), K)
        assert r["accept_len"][b] == j
        assert list(r["out_tokens"][b, :j]) == list(tokens[b, :j])
        assert r["out_tokens"][b, j] == am[b, j]
        assert (r["out_tokens"][b, j + 1:] == -1).all()
    # all draft tokens wrong: exactly one token, the argmax of row 0
    bad = ((am[:, :K] + 1) % V).astype(np.int32)
    r = oracle.verify_linear(target, None, bad, None, np.zeros(B, np.float32), 0.0, lib=oracle_lib)
    assert (r["accept_len"] == 0).all()
    assert (r["out_tokens"][:, 0] == am[:, 0]).all()


def test_tiny_temperature_reduces_to_greedy(oracle_lib):
    """At T -> 0 with draft tokens drawn as a T -> 0 draft would (its argmax),
    speculative sampling is greedy decoding: p/q -> 0 when x misses the target's
    argmax, -> infinity (or 1) when it hits it; the residual and p_K become
    one-hot at the target's argmax."""
    rng = np.random.default_rng(12)
    B, K, V = 30, 4, 50
    base = rng.permutation(np.arange(V, dtype=np.float32))       # distinct, gaps >= 1
    target = np.stack([[rng.permutation(base) for _ in range(K + 1)] for _ in range(B)])
    draft = np.stack([[rng.permutation(base) for _ in range(K)] for _ in range(B)])
    am = target.argmax(-1)
    # a draft sampled at T -> 0 proposes its own argmax; half the time it agrees with the target
    dam = draft.argmax(-1)
    tokens = np.where(rng.random((B, K)) < 0.5, am[:, :K], dam).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    g = oracle.verify_linear(target, None, tokens, None, ub, 0.0, lib=oracle_lib)
    s = oracle.verify_linear(target, draft, tokens, u, ub, 1e-3, lib=oracle_lib)
    np.testing.assert_array_equal(g["accept_len"], s["accept_len"])
    np.testing.assert_array_equal(g["out_tokens"], s["out_tokens"])


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_invariants_random(oracle_lib, dtype):
    rng = np.random.default_rng(13)
    B, K, V, T = 64, 6, 300, 0.8
    t = (2.0 * rng.standard_normal((B, K + 1, V))).astype(np.float32)
    d = (t[:, :K] + 0.7 * rng.standard_normal((B, K, V))).astype(np.float32)
    if dtype == "bf16":
        t = (t.view(np.uint32) >> 16).astype(np.uint16)
        d = (d.view(np.uint32) >> 16).astype(np.uint16)
    tokens = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    r = oracle.verify_linear(t, d, tokens, u, ub, T, lib=oracle_lib)
    j = r["accept_len"]
    assert ((0 <= j) & (j <= K)).all()
    assert (r["num_emitted"] == j + 1).all()                       # at most K + 1, extra always present
    for b in range(B):
        assert list(r["out_tokens"][b, :j[b]]) == list(tokens[b, :j[b]])
        assert 0 <= r["out_tokens"][b, j[b]] < V
        assert (r["out_tokens"][b, j[b] + 1:] == -1).all()
        if j[b] < K:
            # a rejected x has p(x) < q(x), so its residual weight is zero
            assert r["out_tokens"][b, j[b]] != tokens[b, j[b]]
            assert u[b, j[b]] >= r["probs"][b, j[b], 2]
        for i in range(j[b]):
            assert u[b, i] < r["probs"][b, i, 2]
    # without u_bonus: no extra token
    r2 = oracle.verify_linear(t, d, tokens, u, None, T, lib=oracle_lib)
    np.testing.assert_array_equal(r2["accept_len"], j)
    assert (r2["num_emitted"] == j).all()


def test_residual_zero_weight_token_never_drawn(oracle_lib):
    """u_b = 0 must still land on a token of positive residual weight."""
    rng = np.random.default_rng(14)
    B, V = 50, 20
    t = rng.standard_normal((B, 2, V)).astype(np.float32)
    d = rng.standard_normal((B, 1, V)).astype(np.float32)
    r = oracle.sample_bonus(t, d, np.zeros(B, np.int32), np.zeros(B, np.float32), 1.0, lib=oracle_lib)
    for b in range(B):
        p = softmax64(t[b, 0], 1.0)
        q = softmax64(d[b, 0], 1.0)
        w = np.maximum(p - q, 0)
        assert w[r["bonus_token"][b]] > 0
        assert r["bonus_token"][b] == np.nonzero(w > 0)[0][0]


def test_bf16_decoding_equals_fp32_values(oracle_lib):
    rng = np.random.default_rng(15)
    B, K, V = 16, 3, 1000
    bits_t = rng.integers(0, 1 << 16, (B, K + 1, V), dtype=np.uint32).astype(np.uint16)
    bits_d = rng.integers(0, 1 << 16, (B, K, V), dtype=np.uint32).astype(np.uint16)
    # keep finite, moderate values: clear the top exponent bits
    bits_t = (bits_t & 0x81FF) | 0x3C00
    bits_d = (bits_d & 0x81FF) | 0x3C00
    f_t = (bits_t.astype(np.uint32) << 16).view(np.float32)
    f_d = (bits_d.astype(np.uint32) << 16).view(np.float32)
    tokens = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    a = oracle.verify_linear(bits_t, bits_d, tokens, u, ub, 0.9, lib=oracle_lib)
    b = oracle.verify_linear(f_t, f_d, tokens, u, ub, 0.9, lib=oracle_lib)
    for k in ("accept_len", "out_tokens", "num_emitted", "probs", "bonus_cdf"):
        np.testing.assert_array_equal(a[k], b[k])
    # and the decoder maps known bit patterns to known values
    known = np.array([[[0x3F80, 0xC000, 0x4049, 0x0000]]], np.uint16)   # 1, -2, 3.140625, 0
    one = oracle.verify_linear(np.repeat(known, 2, axis=1), None, np.array([[2]], np.int32), None,
                               np.zeros(1, np.float32), 0.0, lib=oracle_lib)
    assert one["accept_len"][0] == 1 and one["out_tokens"][0, 1] == 2


def test_sample_bonus_matches_fused_extra_token(oracle_lib):
    rng = np.random.default_rng(16)
    B, K, V, T = 40, 4, 200, 0.9
    t = (1.5 * rng.standard_normal((B, K + 1, V))).astype(np.float32)
    d = (t[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    tokens = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    r = oracle.verify_linear(t, d, tokens, u, ub, T, lib=oracle_lib)
    s = oracle.sample_bonus(t, d, r["accept_len"], ub, T, lib=oracle_lib)
    j = r["accept_len"]
    np.testing.assert_array_equal(s["bonus_token"], r["out_tokens"][np.arange(B), j])
    np.testing.assert_array_equal(s["bonus_cdf"], r["bonus_cdf"])


def check_strict_acceptance_at_an_exact_ratio(lib):
    """u equal to min(1, p/q) rejects: the test is strict (the reading taken for the cited method).

    V = 4, target logits all 0 (p = 1/4 each), draft logits (0, 0, -inf, -inf) (q = 1/2, 1/2, 0, 0):
    for x = 0 the ratio p/q is exactly 1/2 in binary floating point, and u = 1/2 is exact too."""
    target = np.zeros((2, 2, 4), np.float32)
    draft = np.array([[[0.0, 0.0, -np.inf, -np.inf]]] * 2, np.float32)
    tokens = np.zeros((2, 1), np.int32)
    u = np.array([[0.5], [0.4999999]], np.float32)
    r = oracle.verify_linear(target, draft, tokens, u, None, 1.0, lib=lib)
    assert r["probs"][0, 0, 2] == 0.5
    assert list(r["accept_len"]) == [0, 1]


def check_greedy_rejects_an_out_of_range_token(lib):
    target = np.zeros((3, 3, 5), np.float32)
    target[:, :, 2] = 1.0                       # argmax 2 everywhere
    tokens = np.array([[2, -1], [2, 5], [2, 2]], np.int32)
    r = oracle.verify_linear(target, None, tokens, None, None, 0.0, lib=lib)
    assert list(r["accept_len"]) == [1, 1, 2]


def test_strict_acceptance_at_an_exact_ratio(oracle_lib):
    check_strict_acceptance_at_an_exact_ratio(oracle_lib)


def test_greedy_rejects_an_out_of_range_token(oracle_lib):
    check_greedy_rejects_an_out_of_range_token(oracle_lib)


def check_extra_token_alone_rows_and_lengths(lib):
    """Greedy: the extra token at length j is numpy's argmax of target row j; a length outside
    [0, K] gives -1 (the caller's error, reported by the token)."""
    rng = np.random.default_rng(17)
    B, K, V = 30, 3, 40
    t = rng.integers(-4, 5, (B, K + 1, V)).astype(np.float32)
    al = rng.integers(0, K + 1, B).astype(np.int32)
    al[:3] = [-1, K + 1, K]
    s = oracle.sample_bonus(t, None, al, None, 0.0, lib=lib)
    for b in range(B):
        want = -1 if (al[b] < 0 or al[b] > K) else int(t[b, al[b]].argmax())
        assert s["bonus_token"][b] == want, (b, al[b])


def check_vanished_residual_draws_from_p(lib):
    """Identical target and draft rows leave max(0, p - q) = 0 everywhere: the draw falls back
    to p_j itself (and is flagged), i.e. the first v whose cumulative p exceeds u."""
    rng = np.random.default_rng(18)
    B, K, V, T = 25, 2, 30, 0.8
    t = (2.0 * rng.standard_normal((B, K + 1, V))).astype(np.float32)
    d = t[:, :K].copy()
    al = np.zeros(B, np.int32)
    ub = rng.random(B).astype(np.float32)
    s = oracle.sample_bonus(t, d, al, ub, T, lib=lib)
    assert (s["flags"] & 1).all()
    for b in range(B):
        x = t[b, 0].astype(np.float64) / T
        c = np.cumsum(np.exp(x - x.max()))
        c /= c[-1]
        if np.min(np.abs(c - ub[b])) < 1e-9:
            continue
        assert s["bonus_token"][b] == int(np.searchsorted(c, ub[b], side="right"))


def test_extra_token_alone_rows_and_lengths(oracle_lib):
    check_extra_token_alone_rows_and_lengths(oracle_lib)


def test_vanished_residual_draws_from_p(oracle_lib):
    check_vanished_residual_draws_from_p(oracle_lib)
