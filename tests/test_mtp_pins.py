"""Pins of the oracle's MTP token plug-in.

"Beschleunigung von Sonar durch Spekulation" (Perplexity):
  section "MTP": the draft layer predicts token t_{i+1} from the logits L_i of
    token t_i, which come from the hidden state H_i, so the draft's input token
    buffer is shifted one step left against the target's hidden states;
  section "MTP-Zeitplan für ein einzelnes Token": the target scores 2 * D
    tokens (D sequences); after the target's input tokens are shifted, a kernel
    inserts the target's next tokens at their places, so that no CPU-GPU
    synchronisation follows acceptance; the draft then runs over the same
    positions, doing redundant work on positions that were not accepted.

The pins: hand-worked rows (the page's single-token case and K = 2), the
alignment of every accepted position with the token that follows it in a
list-based simulation of the decoded sequence, the redundant positions, the
lengths, and counts outside [0, K + 1].
"""
import numpy as np

import oracle


def check_hand_worked_single_token(lib):
    # D = 2 sequences, two scored tokens each: (the token the step starts from, the draft token)
    inp = np.array([[100, 7], [200, 8]], np.int32)
    out_tokens = np.array([[7, 31], [12, -1]], np.int32)   # seq 0 accepts 7, extra 31; seq 1 rejects, draws 12
    r = oracle.mtp_plug(inp, out_tokens, [2, 1], pad=0, seq_lens=[50, 60], lib=lib)
    assert r["next_tokens"].tolist() == [[7, 31], [12, 0]]
    assert r["seq_lens"].tolist() == [52, 61] and not r["bad"]


def check_hand_worked_k2(lib):
    inp = np.array([[5, 9, 4], [6, 8, 3], [1, 2, 7]], np.int32)
    out_tokens = np.array([[9, 4, 42], [17, -1, -1], [2, 55, -1]], np.int32)
    r = oracle.mtp_plug(inp, out_tokens, [3, 1, 2], pad=-5, seq_lens=[10, 20, 30], lib=lib)
    assert r["next_tokens"].tolist() == [[9, 4, 42], [17, 3, -5], [2, 55, -5]]
    assert r["seq_lens"].tolist() == [13, 21, 32]


def check_alignment_with_decoded_sequences(lib, K=4, B=64, V=50, seed=3):
    """Position i <= j of the draft's input must hold the token that follows target position i in the
    decoded sequence; later positions are the shifted draft tokens; the length grows by j + 1."""
    rng = np.random.default_rng(seed)
    target = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    draft = (target[:, :K] + 0.7 * rng.standard_normal((B, K, V))).astype(np.float32)
    x = np.array([[rng.choice(V, p=np.exp(r) / np.exp(r).sum()) for r in draft[b]] for b in range(B)], np.int32)
    o = oracle.verify_linear(target, draft, x, rng.random((B, K)).astype(np.float32),
                             rng.random(B).astype(np.float32), 1.0, lib=lib)
    contexts = [list(rng.integers(0, V, size=int(rng.integers(1, 9)))) for _ in range(B)]
    inp = np.array([[c[-1]] + list(x[b]) for b, c in enumerate(contexts)], np.int32)
    lens = np.array([len(c) for c in contexts], np.int32)
    r = oracle.mtp_plug(inp, o["out_tokens"], o["num_emitted"], pad=-1, seq_lens=lens, lib=lib)
    for b, c in enumerate(contexts):
        j = int(o["accept_len"][b])
        decoded = c + list(x[b, :j]) + [int(o["out_tokens"][b, j])]   # the sequence after this step
        L = len(c)
        for i in range(j + 1):          # target position i sits at L - 1 + i; the token after it
            assert r["next_tokens"][b, i] == decoded[L + i]
        for i in range(j + 1, K):       # redundant work: the shifted draft tokens
            assert r["next_tokens"][b, i] == x[b, i]
        if j < K:
            assert r["next_tokens"][b, K] == -1
        assert r["seq_lens"][b] == len(decoded)


def check_nothing_emitted_is_the_shift(lib):
    inp = np.arange(12, dtype=np.int32).reshape(3, 4)
    r = oracle.mtp_plug(inp, np.full((3, 4), 99, np.int32), [0, 0, 0], pad=7, seq_lens=[1, 2, 3], lib=lib)
    assert r["next_tokens"].tolist() == [[1, 2, 3, 7], [5, 6, 7, 7], [9, 10, 11, 7]]
    assert r["seq_lens"].tolist() == [1, 2, 3] and not r["bad"]


def check_counts_out_of_range(lib):
    inp = np.array([[1, 2, 3], [4, 5, 6], [7, 8, 9]], np.int32)
    ot = np.array([[20, 21, 22], [30, 31, 32], [40, 41, 42]], np.int32)
    r = oracle.mtp_plug(inp, ot, [-1, 4, 3], pad=0, seq_lens=[10, 10, 10], lib=lib)
    assert r["bad"]
    assert r["next_tokens"].tolist() == [[2, 3, 0], [5, 6, 0], [40, 41, 42]]
    assert r["seq_lens"].tolist() == [10, 10, 13]


def check_lengths_optional(lib):
    inp = np.array([[1, 2]], np.int32)
    r = oracle.mtp_plug(inp, np.array([[2, 9]], np.int32), [2], pad=0, seq_lens=None, lib=lib)
    assert r["next_tokens"].tolist() == [[2, 9]] and r["seq_lens"] is None


def test_hand_worked_single_token(oracle_lib):
    check_hand_worked_single_token(oracle_lib)


def test_hand_worked_k2(oracle_lib):
    check_hand_worked_k2(oracle_lib)


def test_alignment_with_decoded_sequences(oracle_lib):
    check_alignment_with_decoded_sequences(oracle_lib)
    check_alignment_with_decoded_sequences(oracle_lib, K=1, B=200, seed=4)


def test_nothing_emitted_is_the_shift(oracle_lib):
    check_nothing_emitted_is_the_shift(oracle_lib)


def test_counts_out_of_range(oracle_lib):
    check_counts_out_of_range(oracle_lib)


def test_lengths_optional(oracle_lib):
    check_lengths_optional(oracle_lib)
